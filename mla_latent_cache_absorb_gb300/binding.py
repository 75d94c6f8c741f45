"""ctypes binding to libmla.so: the C ABI of include/mla.h, same names, argument marshalling
only. Pointers may be given as ints, torch tensors (their data_ptr) or None; streams as ints,
torch.cuda.Stream objects or None. Every call returns the library's status code.

The library is required: importing this module without a built libmla.so raises, so the
product path can never fall back to anything else.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_double, c_float, c_int32, c_int64, c_size_t, c_uint64, c_void_p

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmla.so")

MLA_F32, MLA_BF16, MLA_Q8_0, MLA_Q4_AFFINE = 0, 1, 2, 3
STATUS = {
    0: "MLA_OK", 1: "MLA_ERR_INVALID_ARG", 2: "MLA_ERR_UNSUPPORTED", 3: "MLA_ERR_POS_MISMATCH",
    4: "MLA_ERR_CACHE_FULL", 5: "MLA_ERR_WORKSPACE", 6: "MLA_ERR_TIMEOUT", 7: "MLA_ERR_CUDA",
    8: "MLA_ERR_BAD_SEQ_LEN", 9: "MLA_ERR_BAD_PAGE", 10: "MLA_ERR_BAD_KV_B",
}
STATUS_CODE = {v: k for k, v in STATUS.items()}


class MlaConfig(ctypes.Structure):
    _fields_ = [
        ("n_heads", c_int32), ("kv_lora", c_int32), ("qk_nope", c_int32), ("qk_rope", c_int32),
        ("v_head", c_int32), ("act_dtype", c_int32), ("kv_b_dtype", c_int32),
        ("softmax_scale", c_float), ("rms_eps", c_float), ("page_size", c_int32),
        ("max_pages_per_seq", c_int32), ("rows_per_seq", c_int64), ("rope_inv_freq", c_void_p),
    ]


class MlaCache(ctypes.Structure):
    _fields_ = [("rows", c_void_p), ("page_table", c_void_p), ("n_physical_rows", c_int64)]


class MlaProj(ctypes.Structure):
    _fields_ = [("hidden", c_int32), ("q_lora", c_int32), ("w_dtype", c_int32), ("q_norm_eps", c_float),
                ("w_q_a", c_void_p), ("q_a_norm_w", c_void_p), ("w_q", c_void_p), ("w_kva", c_void_p),
                ("w_o", c_void_p)]


class MlaPlanInfo(ctypes.Structure):
    _fields_ = [("kernel", c_int32), ("heads_per_cta", c_int32), ("head_groups", c_int32),
                ("splits", c_int32), ("rows_per_split", c_int64), ("capacity", c_int64)]


if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
_lib = ctypes.CDLL(LIB_PATH)

_CFG = POINTER(MlaConfig)
_CACHE = POINTER(MlaCache)
_PROJ = POINTER(MlaProj)
_SIGS = {
    "mla_status_string": (c_char_p, [c_int32]),
    "mla_abi_version": (c_int32, []),
    "mla_yarn_inv_freq": (c_int32, [c_int32, c_double, c_double, c_int32, c_double, c_double, c_void_p]),
    "mla_yarn_mscale": (c_double, [c_double, c_double]),
    "mla_softmax_scale": (c_float, [c_int32, c_int32, c_double]),
    "mla_validate_kv_b": (c_int32, [c_int32, c_int64, c_int64, c_uint64, c_int32, c_int32, c_int32, c_int32]),
    "mla_kv_b_bytes": (c_uint64, [_CFG]),
    "mla_append_workspace_size": (c_int32, [_CFG, c_int32, POINTER(c_size_t)]),
    "mla_decode_workspace_size": (c_int32, [_CFG, c_int32, POINTER(c_size_t)]),
    "mla_decode_plan": (c_int32, [_CFG, c_int32, POINTER(MlaPlanInfo)]),
    "mla_set_wait_limit_ns": (c_uint64, [c_uint64]),
    "mla_cache_append": (c_int32, [_CFG, _CACHE, c_void_p, c_void_p, c_int32, c_void_p, c_void_p,
                                   c_void_p, c_int32, c_void_p, c_size_t, c_void_p]),
    "mla_decode_attn": (c_int32, [_CFG, c_void_p, c_void_p, _CACHE, c_void_p, c_void_p, c_void_p,
                                  c_void_p, c_int32, c_void_p, c_size_t, c_void_p]),
    "mla_decode_absorb": (c_int32, [_CFG, c_void_p, c_void_p, c_void_p, c_int32, c_void_p, c_size_t, c_void_p]),
    "mla_decode_partial": (c_int32, [_CFG, _CACHE, c_void_p, c_int32, c_void_p, c_size_t, c_void_p]),
    "mla_decode_combine": (c_int32, [_CFG, c_void_p, c_void_p, c_void_p, c_void_p, c_int32, c_void_p,
                                     c_size_t, c_void_p]),
    "mla_get_device_error": (c_int32, [c_void_p, POINTER(c_int32), c_void_p]),
    "mla_clear_device_error": (c_int32, [c_void_p, c_void_p]),
    "mla_decode_attn_noalloc": (c_int32, [_CFG, c_void_p, c_void_p, _CACHE, c_void_p, c_void_p, c_void_p,
                                          c_void_p, c_int32, c_void_p, c_void_p]),
    "mla_front_end_workspace_size": (c_int32, [_CFG, _PROJ, c_int32, POINTER(c_size_t)]),
    "mla_front_end": (c_int32, [_CFG, _PROJ, c_void_p, c_void_p, c_void_p, c_int32, c_void_p, c_size_t,
                                c_void_p]),
    "mla_o_proj_workspace_size": (c_int32, [_CFG, _PROJ, c_int32, POINTER(c_size_t)]),
    "mla_proj_launches": (c_int32, [_CFG, _PROJ, c_int32, POINTER(c_int32), POINTER(c_int32)]),
    "mla_o_proj": (c_int32, [_CFG, _PROJ, c_void_p, c_void_p, c_int32, c_void_p, c_size_t, c_void_p]),
    "mla_decode_multi_workspace_size": (c_int32, [_CFG, c_int32, c_int32, POINTER(c_size_t)]),
    "mla_decode_attn_multi": (c_int32, [_CFG, c_int32, c_void_p, c_void_p, _CACHE, c_void_p, c_void_p, c_void_p,
                                        c_void_p, c_int32, c_void_p, c_size_t, c_void_p]),
}
for _name, (_res, _args) in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.restype = _res
    _f.argtypes = _args

EXPORTED = tuple(_SIGS)


def _p(x):
    """A pointer argument: None, an int address, a torch tensor or a numpy array (host)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if hasattr(x, "ctypes"):
        return x.ctypes.data
    raise TypeError(f"cannot pass {type(x)} as a pointer")


def _s(stream):
    if stream is None:
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class MlaError(RuntimeError):
    def __init__(self, status, where=""):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} ({mla_status_string(status)})")


def check(status, where=""):
    if status != 0:
        raise MlaError(status, where)
    return status


# ---- the C ABI, one wrapper per symbol -----------------------------------------------------

def mla_status_string(s):
    return _lib.mla_status_string(int(s)).decode()


def mla_abi_version():
    return _lib.mla_abi_version()


def mla_yarn_inv_freq(rope_dim, theta, factor, orig_max_pos, beta_fast, beta_slow, out_host):
    return _lib.mla_yarn_inv_freq(rope_dim, theta, factor, orig_max_pos, beta_fast, beta_slow, _p(out_host))


def mla_yarn_mscale(factor, coeff):
    return _lib.mla_yarn_mscale(factor, coeff)


def mla_softmax_scale(qk_nope, qk_rope, mscale):
    return _lib.mla_softmax_scale(qk_nope, qk_rope, mscale)


def mla_validate_kv_b(dtype, rows, cols, size_bytes, heads, nope, kv_lora, v_dim):
    return _lib.mla_validate_kv_b(dtype, rows, cols, size_bytes, heads, nope, kv_lora, v_dim)


def mla_kv_b_bytes(cfg):
    return _lib.mla_kv_b_bytes(ctypes.byref(cfg))


def mla_append_workspace_size(cfg, B):
    n = c_size_t(0)
    st = _lib.mla_append_workspace_size(ctypes.byref(cfg), B, ctypes.byref(n))
    return st, n.value


def mla_decode_workspace_size(cfg, B):
    n = c_size_t(0)
    st = _lib.mla_decode_workspace_size(ctypes.byref(cfg), B, ctypes.byref(n))
    return st, n.value


def mla_decode_plan(cfg, B):
    info = MlaPlanInfo()
    st = _lib.mla_decode_plan(ctypes.byref(cfg), B, ctypes.byref(info))
    return st, info


def mla_set_wait_limit_ns(ns):
    return _lib.mla_set_wait_limit_ns(int(ns))


def mla_cache_append(cfg, cache, kv_in, w_kva, hidden, norm_w, positions, seq_lens, B, workspace,
                     ws_bytes, stream=None):
    return _lib.mla_cache_append(ctypes.byref(cfg), ctypes.byref(cache), _p(kv_in), _p(w_kva), hidden,
                                 _p(norm_w), _p(positions), _p(seq_lens), B, _p(workspace), ws_bytes,
                                 _s(stream))


def mla_decode_attn(cfg, q, kv_b, cache, seq_lens, positions, out, lse, B, workspace, ws_bytes,
                    stream=None):
    return _lib.mla_decode_attn(ctypes.byref(cfg), _p(q), _p(kv_b), ctypes.byref(cache), _p(seq_lens),
                                _p(positions), _p(out), _p(lse), B, _p(workspace), ws_bytes, _s(stream))


def mla_decode_absorb(cfg, q, kv_b, positions, B, workspace, ws_bytes, stream=None):
    return _lib.mla_decode_absorb(ctypes.byref(cfg), _p(q), _p(kv_b), _p(positions), B, _p(workspace),
                                  ws_bytes, _s(stream))


def mla_decode_partial(cfg, cache, seq_lens, B, workspace, ws_bytes, stream=None):
    return _lib.mla_decode_partial(ctypes.byref(cfg), ctypes.byref(cache), _p(seq_lens), B,
                                   _p(workspace), ws_bytes, _s(stream))


def mla_decode_combine(cfg, kv_b, seq_lens, out, lse, B, workspace, ws_bytes, stream=None):
    return _lib.mla_decode_combine(ctypes.byref(cfg), _p(kv_b), _p(seq_lens), _p(out), _p(lse), B,
                                   _p(workspace), ws_bytes, _s(stream))


def mla_get_device_error(workspace, stream=None):
    seq = c_int32(-1)
    st = _lib.mla_get_device_error(_p(workspace), ctypes.byref(seq), _s(stream))
    return st, seq.value


def mla_clear_device_error(workspace, stream=None):
    return _lib.mla_clear_device_error(_p(workspace), _s(stream))


MLA_NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024


def mla_decode_attn_noalloc(cfg, q, kv_b, cache, seq_lens, positions, out, lse, B, device_error=None,
                            stream=None):
    return _lib.mla_decode_attn_noalloc(ctypes.byref(cfg), _p(q), _p(kv_b), ctypes.byref(cache),
                                        _p(seq_lens), _p(positions), _p(out), _p(lse), B,
                                        _p(device_error), _s(stream))


def mla_front_end_workspace_size(cfg, pj, B):
    n = c_size_t(0)
    st = _lib.mla_front_end_workspace_size(ctypes.byref(cfg), ctypes.byref(pj), B, ctypes.byref(n))
    return st, n.value


def mla_front_end(cfg, pj, x, q, kva, B, workspace, ws_bytes, stream=None):
    return _lib.mla_front_end(ctypes.byref(cfg), ctypes.byref(pj), _p(x), _p(q), _p(kva), B, _p(workspace),
                              ws_bytes, _s(stream))


def mla_o_proj_workspace_size(cfg, pj, B):
    n = c_size_t(0)
    st = _lib.mla_o_proj_workspace_size(ctypes.byref(cfg), ctypes.byref(pj), B, ctypes.byref(n))
    return st, n.value


def mla_proj_launches(cfg, pj, B):
    """(status, kernels of one mla_front_end call, kernels of one mla_o_proj call)."""
    fe, op = c_int32(0), c_int32(0)
    st = _lib.mla_proj_launches(ctypes.byref(cfg), ctypes.byref(pj), B, ctypes.byref(fe), ctypes.byref(op))
    return st, fe.value, op.value


def mla_o_proj(cfg, pj, attn, y, B, workspace, ws_bytes, stream=None):
    return _lib.mla_o_proj(ctypes.byref(cfg), ctypes.byref(pj), _p(attn), _p(y), B, _p(workspace), ws_bytes,
                           _s(stream))


def mla_decode_multi_workspace_size(cfg, tokens, B):
    n = c_size_t(0)
    st = _lib.mla_decode_multi_workspace_size(ctypes.byref(cfg), tokens, B, ctypes.byref(n))
    return st, n.value


def mla_decode_attn_multi(cfg, tokens, q, kv_b, cache, seq_lens, positions, out, lse, B, workspace, ws_bytes,
                          stream=None):
    return _lib.mla_decode_attn_multi(ctypes.byref(cfg), tokens, _p(q), _p(kv_b), ctypes.byref(cache),
                                      _p(seq_lens), _p(positions), _p(out), _p(lse), B, _p(workspace), ws_bytes,
                                      _s(stream))
