"""Device-side set-up of one step through the C ABI, with PyTorch as the allocator.

`DeviceStep` uploads a synthetic problem (see `synth`), builds the `mla_config` /
`mla_cache` structs, sizes and clears the workspaces, and runs the two calls of the step:
`mla_cache_append` then `mla_decode_attn`. Every step of the method runs in libmla's
kernels; torch only owns memory and streams.
"""
from __future__ import annotations

import numpy as np
import torch

from . import binding as L

_DT = {"f32": L.MLA_F32, "bf16": L.MLA_BF16, "q8_0": L.MLA_Q8_0, "q4_affine": L.MLA_Q4_AFFINE}


def _dev(a: np.ndarray, device) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to(device)


def make_config(wl, inv_freq_dev: torch.Tensor, rows_per_seq: int, max_pages: int) -> L.MlaConfig:
    """mla_config for a workload; the softmax scale and YaRN table come from the library's
    host helpers."""
    mscale = L.mla_yarn_mscale(wl.yarn_factor, wl.yarn_mscale_coeff)
    cfg = L.MlaConfig()
    cfg.n_heads, cfg.kv_lora, cfg.qk_nope, cfg.qk_rope, cfg.v_head = wl.H, wl.C, wl.N, wl.R, wl.V
    cfg.act_dtype = _DT[wl.act]
    cfg.kv_b_dtype = _DT[wl.kv_b]
    cfg.softmax_scale = L.mla_softmax_scale(wl.N, wl.R, mscale)
    cfg.rms_eps = wl.rms_eps
    cfg.page_size = wl.page_size
    cfg.max_pages_per_seq = max_pages
    cfg.rows_per_seq = rows_per_seq
    cfg.rope_inv_freq = inv_freq_dev.data_ptr()
    return cfg


def yarn_table(wl, device) -> torch.Tensor:
    host = np.zeros(wl.R // 2, dtype=np.float64)
    L.check(L.mla_yarn_inv_freq(wl.R, wl.rope_theta, wl.yarn_factor, wl.yarn_orig_max_pos,
                                wl.yarn_beta_fast, wl.yarn_beta_slow, host), "mla_yarn_inv_freq")
    return torch.from_numpy(host).to(device)


class DeviceStep:
    """One problem resident on the GPU, ready to run append + decode through the C ABI."""

    def __init__(self, prob, device="cuda:0", stream=None):
        wl = prob.wl
        self.prob, self.wl, self.device = prob, wl, torch.device(device)
        self.stream = stream if stream is not None else torch.cuda.current_stream(self.device)
        d = self.device
        self.inv_freq = yarn_table(wl, d)
        self.cfg = make_config(wl, self.inv_freq, prob.rows_per_seq, prob.max_pages)
        self.q = _dev(prob.q, d)
        self.pool = _dev(prob.pool, d)
        self.page_table = _dev(prob.page_table, d) if prob.page_table is not None else None
        self.cache = L.MlaCache()
        self.cache.rows = self.pool.data_ptr()
        self.cache.page_table = self.page_table.data_ptr() if self.page_table is not None else None
        self.cache.n_physical_rows = prob.pool.shape[0]
        self.positions = _dev(prob.positions, d)
        self.len_before = _dev(prob.positions, d)       # append writes at the current length
        self.seq_lens = _dev(prob.seq_lens, d)          # rows attended after the append
        self.norm_w = _dev(prob.norm_w, d)
        self.kv_b = _dev(prob.kv_b, d)
        L.check(0 if L.mla_kv_b_bytes(self.cfg) == self.kv_b.numel() * self.kv_b.element_size() else 10,
                "kv_b size")
        if prob.kva_rows is not None:
            self.kv_in, self.w_kva, self.hidden = _dev(prob.kva_rows, d), None, 0
        else:
            self.kv_in, self.w_kva, self.hidden = _dev(prob.x, d), _dev(prob.w_kva, d), wl.hidden
        B = wl.B
        st, n = L.mla_append_workspace_size(self.cfg, B)
        L.check(st, "mla_append_workspace_size")
        self.ws_append = torch.zeros(n, dtype=torch.uint8, device=d)
        st, n = L.mla_decode_workspace_size(self.cfg, B)
        L.check(st, "mla_decode_workspace_size")
        self.ws_decode = torch.zeros(n, dtype=torch.uint8, device=d)
        self.out = torch.empty((B, wl.H, wl.V), dtype=torch.float32, device=d)
        self.lse = torch.empty((B, wl.H), dtype=torch.float32, device=d)

    # ---- the two calls ------------------------------------------------------------------
    def append(self, stream=None):
        s = stream if stream is not None else self.stream
        return L.mla_cache_append(self.cfg, self.cache, self.kv_in, self.w_kva, self.hidden, self.norm_w,
                                  self.positions, self.len_before, self.wl.B, self.ws_append,
                                  self.ws_append.numel(), s)

    def decode(self, stream=None, positions=True):
        s = stream if stream is not None else self.stream
        return L.mla_decode_attn(self.cfg, self.q, self.kv_b, self.cache, self.seq_lens,
                                 self.positions if positions else None, self.out, self.lse, self.wl.B,
                                 self.ws_decode, self.ws_decode.numel(), s)

    def step(self, stream=None):
        L.check(self.append(stream), "mla_cache_append")
        L.check(self.decode(stream), "mla_decode_attn")

    # ---- stages (for timing) ---------------------------------------------------------------
    def absorb(self, stream=None):
        return L.mla_decode_absorb(self.cfg, self.q, self.kv_b, self.positions, self.wl.B, self.ws_decode,
                                   self.ws_decode.numel(), stream if stream is not None else self.stream)

    def partial(self, stream=None):
        return L.mla_decode_partial(self.cfg, self.cache, self.seq_lens, self.wl.B, self.ws_decode,
                                    self.ws_decode.numel(), stream if stream is not None else self.stream)

    def combine(self, stream=None):
        return L.mla_decode_combine(self.cfg, self.kv_b, self.seq_lens, self.out, self.lse, self.wl.B,
                                    self.ws_decode, self.ws_decode.numel(),
                                    stream if stream is not None else self.stream)

    def device_errors(self):
        return (L.mla_get_device_error(self.ws_append, self.stream),
                L.mla_get_device_error(self.ws_decode, self.stream))

    def pool_host(self) -> np.ndarray:
        a = self.pool.cpu().numpy()
        return a.view(np.uint16) if self.wl.act == "bf16" else a
