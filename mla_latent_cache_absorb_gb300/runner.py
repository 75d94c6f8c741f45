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
        T = wl.tokens
        st, n = L.mla_decode_multi_workspace_size(self.cfg, T, B)
        L.check(st, "mla_decode_multi_workspace_size")
        self.ws_decode = torch.zeros(n, dtype=torch.uint8, device=d)
        tok = () if T == 1 else (T,)
        self.out = torch.empty((B,) + tok + (wl.H, wl.V), dtype=torch.float32, device=d)
        self.lse = torch.empty((B,) + tok + (wl.H,), dtype=torch.float32, device=d)

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

    def decode_multi(self, stream=None, positions=True):
        """mla_decode_attn_multi over the workload's query tokens (every row already cached)."""
        s = stream if stream is not None else self.stream
        return L.mla_decode_attn_multi(self.cfg, self.wl.tokens, self.q, self.kv_b, self.cache, self.seq_lens,
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


class DeviceProj:
    """The layer's projections of one problem resident on the GPU: `front_end()` runs
    mla_front_end (q and the kv_a rows) and `o_proj()` runs mla_o_proj, through the C ABI."""

    def __init__(self, pp, device="cuda:0", stream=None, with_kva=True):
        wl = pp.wl
        self.pp, self.wl, self.device = pp, wl, torch.device(device)
        self.stream = stream if stream is not None else torch.cuda.current_stream(self.device)
        d = self.device
        cfg = L.MlaConfig()
        cfg.n_heads, cfg.kv_lora, cfg.qk_nope, cfg.qk_rope, cfg.v_head = wl.H, wl.C, wl.N, wl.R, wl.V
        cfg.act_dtype = _DT[wl.act]
        cfg.kv_b_dtype = L.MLA_BF16
        cfg.softmax_scale = L.mla_softmax_scale(wl.N, wl.R, 1.0)
        cfg.rms_eps = 1e-6
        cfg.page_size, cfg.max_pages_per_seq, cfg.rows_per_seq = 0, 0, 1
        self.cfg = cfg
        self.x = _dev(pp.x, d)
        self.w_q_a = _dev(pp.w_q_a, d) if pp.w_q_a is not None else None
        self.q_a_norm_w = _dev(pp.q_a_norm_w, d) if pp.q_a_norm_w is not None else None
        self.w_q = _dev(pp.w_q, d)
        self.w_kva = _dev(pp.w_kva, d)
        self.w_o = _dev(pp.w_o, d)
        self.attn = _dev(pp.attn, d)
        pj = L.MlaProj()
        pj.hidden, pj.q_lora, pj.w_dtype, pj.q_norm_eps = wl.hidden, wl.q_lora, _DT[wl.w], wl.eps
        pj.w_q_a = self.w_q_a.data_ptr() if self.w_q_a is not None else None
        pj.q_a_norm_w = self.q_a_norm_w.data_ptr() if self.q_a_norm_w is not None else None
        pj.w_q = self.w_q.data_ptr()
        pj.w_kva = self.w_kva.data_ptr() if with_kva else None
        pj.w_o = self.w_o.data_ptr()
        self.pj = pj
        B = wl.B
        act = torch.int16 if wl.act == "bf16" else torch.float32
        self.q = torch.zeros((B, wl.H, wl.N + wl.R), dtype=act, device=d)
        self.kva = torch.zeros((B, wl.C + wl.R), dtype=torch.float32, device=d) if with_kva else None
        self.y = torch.zeros((B, wl.hidden), dtype=torch.float32, device=d)
        st, n = L.mla_front_end_workspace_size(cfg, pj, B)
        L.check(st, "mla_front_end_workspace_size")
        self.ws = torch.zeros(max(n, 256), dtype=torch.uint8, device=d)
        st, n = L.mla_o_proj_workspace_size(cfg, pj, B)
        L.check(st, "mla_o_proj_workspace_size")
        self.ws_o = torch.zeros(max(n, 256), dtype=torch.uint8, device=d)

    def front_end(self, stream=None):
        return L.mla_front_end(self.cfg, self.pj, self.x, self.q, self.kva, self.wl.B, self.ws,
                               self.ws.numel(), self.stream if stream is None else stream)

    def o_proj(self, attn=None, stream=None):
        return L.mla_o_proj(self.cfg, self.pj, self.attn if attn is None else attn, self.y, self.wl.B, self.ws_o,
                            self.ws_o.numel(), self.stream if stream is None else stream)

    def launches(self) -> int:
        """Kernels one front_end() plus one o_proj() enqueue."""
        st, fe, op = L.mla_proj_launches(self.cfg, self.pj, self.wl.B)
        L.check(st, "mla_proj_launches")
        return fe + op

    def q_host(self) -> np.ndarray:
        q = self.q.cpu().numpy()
        return q.view(np.uint16) if self.wl.act == "bf16" else q
