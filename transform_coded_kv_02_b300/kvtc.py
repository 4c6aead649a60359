"""Python binding of libkvtc (transform-coded KV cache for B300 / sm_103a).

Argument marshalling only: every step of calibration, encoding and decode attention runs inside the
C-ABI library (host C++ for calibration, CUDA kernels for the rest). Device buffers are passed as
torch tensors (their data_ptr()) or raw integer addresses; host arrays as numpy arrays. The library must
have been built (python -m transform_coded_kv_02_b300.build); importing fails loudly otherwise.
"""
from __future__ import annotations

import ctypes
import os
import re

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libkvtc.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "kvtc.h")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"libkvtc.so not built at {LIB_PATH}; run: python -m transform_coded_kv_02_b300.build")
_lib = ctypes.CDLL(LIB_PATH)

KV_OK, KV_ERR_INVALID_ARG, KV_ERR_UNSUPPORTED, KV_ERR_BUDGET, KV_ERR_NUMERIC, KV_ERR_CUDA, \
    KV_ERR_TIMEOUT, KV_ERR_IO, KV_ERR_DEVICE = range(9)
STATUS_NAMES = {0: "KV_OK", 1: "KV_ERR_INVALID_ARG", 2: "KV_ERR_UNSUPPORTED", 3: "KV_ERR_BUDGET",
                4: "KV_ERR_NUMERIC", 5: "KV_ERR_CUDA", 6: "KV_ERR_TIMEOUT", 7: "KV_ERR_IO", 8: "KV_ERR_DEVICE"}
KV_DTYPE_F32, KV_DTYPE_BF16 = 0, 1
KV_TENSOR_K, KV_TENSOR_V = 0, 1

c_int, c_int64, c_float, c_void_p, c_size_t = ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t


class kv_calib_set(ctypes.Structure):
    _fields_ = [("k", c_void_p), ("v", c_void_p), ("q", c_void_p), ("n_tok", c_int64), ("n_q", c_int64)]


class kv_calib_opts(ctypes.Structure):
    _fields_ = [("d", c_int), ("bits_k", c_float), ("bits_v", c_float), ("max_bits", c_int), ("n_threads", c_int),
                ("joint", c_int), ("key_basis", c_int)]


class kv_cache(ctypes.Structure):
    _fields_ = [("k_rec", c_void_p), ("v_rec", c_void_p), ("B", c_int), ("Hkv", c_int), ("T_cap", c_int64),
                ("per_seq_params", c_int)]


class kv_paged_cache(ctypes.Structure):
    _fields_ = [("k_pages", c_void_p), ("v_pages", c_void_p), ("n_pages", c_int64), ("page_tokens", c_int),
                ("Hkv", c_int), ("B", c_int), ("n_layers", c_int), ("max_pages", c_int), ("block_table", c_void_p),
                ("per_seq_params", c_int), ("first_layer", c_int)]


def _sig(name, res, args):
    f = getattr(_lib, name)
    f.restype = res
    f.argtypes = args
    return f


_P = c_void_p
_sig("kv_calibrate", c_int, [c_int, ctypes.POINTER(kv_calib_set), ctypes.POINTER(kv_calib_opts), ctypes.POINTER(_P)])
_sig("kv_params_from_arrays", c_int, [c_int, c_int, _P, _P, _P, _P, c_int, _P, _P, _P, _P, c_int, ctypes.POINTER(_P)])
_sig("kv_params_set_inverse", c_int, [_P, c_int, _P])
_sig("kv_params_get_inverse", c_int, [_P, c_int, c_int, _P])
_sig("kv_params_upload", c_int, [_P, _P])
_sig("kv_params_set_rope", c_int, [_P, ctypes.c_double])
_sig("kv_params_get_rope", ctypes.c_double, [_P])
_sig("kv_paged_cache_bytes", c_size_t, [_P, c_int, c_int64, c_int, c_int])
_sig("kv_encode_paged", c_int, [_P, ctypes.POINTER(kv_paged_cache), _P, _P, c_int, c_int64, _P, _P])
_sig("kv_decode_paged_workspace_bytes", c_size_t, [_P, ctypes.POINTER(kv_paged_cache), c_int])
_sig("kv_attend_decode_paged", c_int, [_P, ctypes.POINTER(kv_paged_cache), _P, c_int, _P, _P, c_float, _P, _P,
                                       c_size_t, _P])
_sig("kv_params_num_sets", c_int, [_P])
_sig("kv_params_record_words", c_int, [_P, c_int])
_sig("kv_params_info", c_int, [_P, c_int, c_int, _P, _P, _P, _P, _P, _P])
_sig("kv_params_save", c_int, [_P, ctypes.c_char_p])
_sig("kv_params_load", c_int, [ctypes.c_char_p, ctypes.POINTER(_P)])
_sig("kv_params_free", None, [_P])
_sig("kv_cache_bytes", c_size_t, [_P, c_int, c_int, c_int, c_int64])
_sig("kv_encode", c_int, [_P, ctypes.POINTER(kv_cache), _P, _P, c_int, c_int, c_int64, _P, _P])
_sig("kv_decode_workspace_bytes", c_size_t, [_P, c_int, c_int, c_int, c_int64])
_sig("kv_attend_decode", c_int, [_P, ctypes.POINTER(kv_cache), _P, c_int, c_int, _P, c_float, _P, _P, c_size_t, _P])
_sig("kv_attend_decode_noalloc", c_int, [_P, ctypes.POINTER(kv_cache), _P, c_int, c_int, _P, c_float, _P, _P])
_sig("kv_token_weights_workspace_bytes", c_size_t, [c_int, c_int, c_int64])
_sig("kv_token_weights", c_int, [_P, c_int, _P, c_int, c_int, c_int, c_int64, c_float, _P, _P, c_size_t, _P])
_sig("kv_token_select", c_int, [_P, c_int, c_int, c_int64, c_int64, _P, _P])
_sig("kv_cache_compact", c_int, [_P, ctypes.POINTER(kv_cache), ctypes.POINTER(kv_cache), c_int, _P, c_int64, _P])
_sig("kv_decode_bf16_workspace_bytes", c_size_t, [c_int, c_int, c_int, c_int64])
_sig("kv_attend_decode_bf16", c_int, [_P, _P, c_int, c_int, c_int, c_int64, _P, _P, c_float, _P, _P, c_size_t, _P])
_sig("kv_check_status", c_int, [_P])
_sig("kv_last_error", ctypes.c_char_p, [])
_sig("kv_version", c_int, [])
_sig("kv_debug_quantize_pack", c_int, [_P, c_int, c_int, _P, c_int64, _P, c_int, _P])
_sig("kv_debug_unpack", c_int, [_P, c_int, c_int, _P, c_int64, _P, _P])
_sig("kv_debug_water_fill", c_int, [_P, c_int, c_int, c_int, _P])
_sig("kv_debug_eigh", c_int, [_P, c_int, _P, _P])
_sig("kv_debug_set_encode_path", c_int, [c_int])
_sig("kv_debug_set_wait_limit_ns", c_int, [ctypes.c_longlong])
_sig("kv_debug_wait_timeout_selftest", c_int, [_P])
_sig("kv_debug_decode_plan", c_int, [_P, c_int, c_int, c_int, ctypes.c_int64, _P])


class KvError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn}: {STATUS_NAMES.get(status, status)}: {_lib.kv_last_error().decode()}")


def _check(fn, st):
    if st != KV_OK:
        raise KvError(fn, st)


def _ptr(x):
    """Address of a device buffer (torch tensor / int) or a host numpy array."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    raise TypeError(type(x))


_torch = None  # the torch module once looked up (False when it is not installed)


def _stream(stream):
    if stream is None:
        global _torch
        if _torch is None:
            try:
                import torch
                _torch = torch
            except ImportError:
                _torch = False
        # before CUDA is initialised in this process the current stream is the default stream
        if _torch and _torch.cuda.is_initialized():
            return _torch.cuda.current_stream().cuda_stream
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def exported_symbols():
    """Function names declared in include/kvtc.h."""
    text = open(HEADER_PATH).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kv_[a-z0-9_]+)\s*\(", text)))


# ------------------------------------------------------------------------------------------------------
class Params:
    """Owner of a kv_params* (freed on garbage collection)."""

    def __init__(self, handle):
        self.handle = handle

    def __del__(self):
        if getattr(self, "handle", None):
            _lib.kv_params_free(self.handle)
            self.handle = None

    @property
    def num_sets(self):
        return _lib.kv_params_num_sets(self.handle)

    def record_words(self, tensor):
        return _lib.kv_params_record_words(self.handle, tensor)

    def upload(self, stream=None):
        _check("kv_params_upload", _lib.kv_params_upload(self.handle, _stream(stream)))
        return self

    def inverse(self, set_idx, tensor, d=128):
        """The stored inverse of one set's transform [d, d], or None for an orthogonal transform."""
        out = np.zeros((d, d), np.float32)
        st = _lib.kv_params_get_inverse(self.handle, set_idx, tensor, _ptr(out))
        if st == KV_ERR_UNSUPPORTED:
            return None
        _check("kv_params_get_inverse", st)
        return out

    def set_inverse(self, tensor, Tinv):
        """A non-orthogonal transform's inverse for tensor 0 (keys) or 1 (values): [S, d, d], Tinv[k][j] with
        column j pairing with storage channel j; None removes it. Takes effect at the next upload."""
        if Tinv is None:
            _check("kv_params_set_inverse", _lib.kv_params_set_inverse(self.handle, tensor, None))
        else:
            a = np.ascontiguousarray(Tinv, np.float32)
            _check("kv_params_set_inverse", _lib.kv_params_set_inverse(self.handle, tensor, _ptr(a)))
        return self

    def set_rope(self, base):
        """Rotary embedding of the decode's queries (pairs (i, i + d/2), angle pos * base^(-2i/d)); 0 removes it.
        Takes effect at the next upload."""
        _check("kv_params_set_rope", _lib.kv_params_set_rope(self.handle, float(base)))
        return self

    @property
    def rope_base(self):
        return _lib.kv_params_get_rope(self.handle)

    def info(self, set_idx, tensor, d=128):
        w = np.zeros(d, np.int32)
        ev = np.zeros(d, np.float64)
        imp = np.zeros(d, np.float64)
        T = np.zeros((d, d), np.float32)
        mu = np.zeros(d, np.float32)
        sg = np.zeros(d, np.float32)
        _check("kv_params_info", _lib.kv_params_info(self.handle, set_idx, tensor, _ptr(w), _ptr(ev), _ptr(imp),
                                                     _ptr(T), _ptr(mu), _ptr(sg)))
        return dict(widths=w, eigvals=ev, importance=imp, T=T, mu=mu, sigma=sg,
                    r_words=self.record_words(tensor))

    def save(self, path):
        _check("kv_params_save", _lib.kv_params_save(self.handle, path.encode()))


def kv_calibrate(sets, bits_k, bits_v, max_bits=8, n_threads=0, d=128, joint=False, attention_aware_keys=False,
                 whitened_keys=False):
    """sets: list of (k [n, d], v [n, d], q [m, d]) host arrays (converted to contiguous fp32); joint: split the
    record words between keys and values jointly instead of by bits_k and bits_v; attention_aware_keys: the
    attention-aware orthogonal key basis instead of the KLT; whitened_keys: the non-orthogonal key transform
    (key_basis 2)."""
    keep = []
    arr = (kv_calib_set * len(sets))()
    for i, (k, v, q) in enumerate(sets):
        k = np.ascontiguousarray(k, np.float32)
        v = np.ascontiguousarray(v, np.float32)
        q = np.ascontiguousarray(q, np.float32)
        keep += [k, v, q]
        arr[i] = kv_calib_set(_ptr(k), _ptr(v), _ptr(q), k.shape[0], q.shape[0])
    opts = kv_calib_opts(d, bits_k, bits_v, max_bits, n_threads, int(joint),
                         2 if whitened_keys else int(attention_aware_keys))
    h = c_void_p()
    _check("kv_calibrate", _lib.kv_calibrate(len(sets), arr, ctypes.byref(opts), ctypes.byref(h)))
    return Params(h.value)


def kv_params_from_arrays(T_k, mu_k, sigma_k, widths_k, r_words_k, T_v, mu_v, sigma_v, widths_v, r_words_v, d=128,
                          T_inv_k=None):
    """Arrays with a leading set axis: T [S, d, d], mu/sigma [S, d], widths [S, d]; T_inv_k [S, d, d]: the key
    transform's inverse when it is not orthogonal."""
    a = [np.ascontiguousarray(x, t) for x, t in ((T_k, np.float32), (mu_k, np.float32), (sigma_k, np.float32),
                                                 (widths_k, np.int32), (T_v, np.float32), (mu_v, np.float32),
                                                 (sigma_v, np.float32), (widths_v, np.int32))]
    S = a[0].shape[0]
    h = c_void_p()
    _check("kv_params_from_arrays", _lib.kv_params_from_arrays(
        d, S, _ptr(a[0]), _ptr(a[1]), _ptr(a[2]), _ptr(a[3]), r_words_k, _ptr(a[4]), _ptr(a[5]), _ptr(a[6]),
        _ptr(a[7]), r_words_v, ctypes.byref(h)))
    P = Params(h.value)
    if T_inv_k is not None:
        P.set_inverse(0, T_inv_k)
    return P


def kv_params_load(path):
    h = c_void_p()
    _check("kv_params_load", _lib.kv_params_load(path.encode(), ctypes.byref(h)))
    return Params(h.value)


def make_cache(k_rec, v_rec, B, Hkv, T_cap, per_seq_params=False):
    return kv_cache(_ptr(k_rec), _ptr(v_rec), B, Hkv, T_cap, int(bool(per_seq_params)))


def kv_cache_bytes(params, tensor, B, Hkv, T_cap):
    return _lib.kv_cache_bytes(params.handle, tensor, B, Hkv, T_cap)


def kv_encode(params, cache, k, v, dtype, B, t_new, dst_pos, stream=None):
    _check("kv_encode", _lib.kv_encode(params.handle, ctypes.byref(cache), _ptr(k), _ptr(v), dtype, B, t_new,
                                       _ptr(dst_pos), _stream(stream)))


def kv_decode_workspace_bytes(params, B, Hkv, Hq, T_cap):
    return _lib.kv_decode_workspace_bytes(params.handle, B, Hkv, Hq, T_cap)


def kv_attend_decode(params, cache, q, B, Hq, seq_lens, softmax_scale, out, workspace, ws_bytes=None, stream=None):
    nbytes = ws_bytes if ws_bytes is not None else workspace.numel() * workspace.element_size()
    _check("kv_attend_decode", _lib.kv_attend_decode(params.handle, ctypes.byref(cache), _ptr(q), B, Hq,
                                                     _ptr(seq_lens), softmax_scale, _ptr(out), _ptr(workspace),
                                                     nbytes, _stream(stream)))


NOALLOC_SCRATCH_BYTES = 4 << 20


def kv_attend_decode_noalloc(params, cache, q, B, Hq, seq_lens, softmax_scale, out, stream=None):
    """Decode attention using the library's fixed static scratch instead of a caller workspace (for callers
    that cannot allocate device memory). Calls that overlap on the GPU race on that scratch."""
    _check("kv_attend_decode_noalloc", _lib.kv_attend_decode_noalloc(params.handle, ctypes.byref(cache), _ptr(q), B,
                                                                     Hq, _ptr(seq_lens), softmax_scale, _ptr(out),
                                                                     _stream(stream)))


def make_paged_cache(k_pages, v_pages, n_pages, page_tokens, Hkv, B, n_layers, max_pages, block_table,
                     per_seq_params=False, first_layer=0):
    """A paged view: pools [n_pages][Hkv][page_tokens][R] (values [n_pages][Hkv][page_tokens / 2][2 R]) and the
    block table [n_layers * B][max_pages] (device int32)."""
    return kv_paged_cache(_ptr(k_pages), _ptr(v_pages), n_pages, page_tokens, Hkv, B, n_layers, max_pages,
                          _ptr(block_table), int(bool(per_seq_params)), first_layer)


def kv_paged_cache_bytes(params, tensor, n_pages, page_tokens, Hkv):
    return _lib.kv_paged_cache_bytes(params.handle, tensor, n_pages, page_tokens, Hkv)


def kv_encode_paged(params, cache, k, v, dtype, t_new, dst_pos, stream=None):
    """k, v: [n_layers][B][Hkv][t_new][d] device arrays; dst_pos: device int64 [B]."""
    _check("kv_encode_paged", _lib.kv_encode_paged(params.handle, ctypes.byref(cache), _ptr(k), _ptr(v), dtype,
                                                   t_new, _ptr(dst_pos), _stream(stream)))


def kv_decode_paged_workspace_bytes(params, cache, Hq):
    return _lib.kv_decode_paged_workspace_bytes(params.handle, ctypes.byref(cache), Hq)


def kv_attend_decode_paged(params, cache, q, Hq, seq_lens, q_pos, softmax_scale, out, workspace, ws_bytes=None,
                           stream=None):
    """q: bf16 [n_layers][B][Hq][d]; out: fp32 likewise; seq_lens: int32 [B]; q_pos: int32 [B] (rotary embedding
    of q in the kernel) or None."""
    nbytes = ws_bytes if ws_bytes is not None else workspace.numel() * workspace.element_size()
    _check("kv_attend_decode_paged", _lib.kv_attend_decode_paged(
        params.handle, ctypes.byref(cache), _ptr(q), Hq, _ptr(seq_lens), None if q_pos is None else _ptr(q_pos),
        softmax_scale, _ptr(out), _ptr(workspace), nbytes, _stream(stream)))


def kv_token_weights_workspace_bytes(B, Hkv, T):
    return _lib.kv_token_weights_workspace_bytes(B, Hkv, T)


def kv_token_weights(q_obs, W, k, B, Hkv, Hq, T, softmax_scale, weights, workspace, ws_bytes=None, stream=None):
    """q_obs: bf16 [B][Hq][W][d]; k: bf16 [B][Hkv][T][d]; weights: fp32 [B][Hkv][T] (device arrays)."""
    nbytes = ws_bytes if ws_bytes is not None else workspace.numel() * workspace.element_size()
    _check("kv_token_weights", _lib.kv_token_weights(_ptr(q_obs), W, _ptr(k), B, Hkv, Hq, T, softmax_scale,
                                                     _ptr(weights), _ptr(workspace), nbytes, _stream(stream)))


def kv_token_select(weights, B, Hkv, T, keep, keep_idx, stream=None):
    """keep_idx: int32 [B][Hkv][keep] (device) receives the kept tokens' indices, ascending."""
    _check("kv_token_select", _lib.kv_token_select(_ptr(weights), B, Hkv, T, keep, _ptr(keep_idx), _stream(stream)))


def kv_cache_compact(params, src, dst, B, keep_idx, keep, stream=None):
    _check("kv_cache_compact", _lib.kv_cache_compact(params.handle, ctypes.byref(src), ctypes.byref(dst), B,
                                                     _ptr(keep_idx), keep, _stream(stream)))


def kv_decode_bf16_workspace_bytes(B, Hkv, Hq, T_cap):
    return _lib.kv_decode_bf16_workspace_bytes(B, Hkv, Hq, T_cap)


def kv_attend_decode_bf16(k, v, B, Hkv, Hq, T_cap, q, seq_lens, softmax_scale, out, workspace, ws_bytes=None,
                          stream=None):
    nbytes = ws_bytes if ws_bytes is not None else workspace.numel() * workspace.element_size()
    _check("kv_attend_decode_bf16", _lib.kv_attend_decode_bf16(_ptr(k), _ptr(v), B, Hkv, Hq, T_cap, _ptr(q),
                                                               _ptr(seq_lens), softmax_scale, _ptr(out),
                                                               _ptr(workspace), nbytes, _stream(stream)))


def kv_check_status(stream=None):
    """Returns the status code (does not raise)."""
    return _lib.kv_check_status(_stream(stream))


def kv_last_error():
    return _lib.kv_last_error().decode()


def kv_version():
    return _lib.kv_version()


def kv_debug_quantize_pack(params, set_idx, tensor, y, n, rec, variant=0, stream=None):
    _check("kv_debug_quantize_pack", _lib.kv_debug_quantize_pack(params.handle, set_idx, tensor, _ptr(y), n,
                                                                 _ptr(rec), variant, _stream(stream)))


def kv_debug_unpack(params, set_idx, tensor, rec, n, codes, stream=None):
    _check("kv_debug_unpack", _lib.kv_debug_unpack(params.handle, set_idx, tensor, _ptr(rec), n, _ptr(codes),
                                                   _stream(stream)))


def kv_debug_water_fill(lam, budget_bits, max_bits=8):
    lam = np.ascontiguousarray(lam, np.float64)
    out = np.zeros(lam.shape[0], np.int32)
    _check("kv_debug_water_fill", _lib.kv_debug_water_fill(_ptr(lam), lam.shape[0], budget_bits, max_bits, _ptr(out)))
    return out


def kv_debug_eigh(sym):
    sym = np.ascontiguousarray(sym, np.float64)
    d = sym.shape[0]
    ev = np.zeros(d)
    vec = np.zeros((d, d))
    _check("kv_debug_eigh", _lib.kv_debug_eigh(_ptr(sym), d, _ptr(ev), _ptr(vec)))
    return ev, vec


def kv_debug_set_encode_path(path):
    _check("kv_debug_set_encode_path", _lib.kv_debug_set_encode_path(path))


def kv_debug_set_wait_limit_ns(ns):
    _check("kv_debug_set_wait_limit_ns", _lib.kv_debug_set_wait_limit_ns(ns))


def kv_debug_decode_plan(params, B, Hkv, Hq, T_cap):
    """The decode launch plan (see include/kvtc.h) as a dict."""
    info = (ctypes.c_int32 * 12)()
    _check("kv_debug_decode_plan", _lib.kv_debug_decode_plan(params.handle, B, Hkv, Hq, T_cap, info))
    v = list(info)
    return {"cluster": v[0], "splits": v[1], "stages": v[2], "warps": v[3], "channel_blocks": v[4],
            "smem_bytes": v[5], "clusters_held": dict(zip((16, 8, 4, 2, 1), v[6:11])), "single_word": v[11]}


def kv_debug_wait_timeout_selftest(stream=None):
    _check("kv_debug_wait_timeout_selftest", _lib.kv_debug_wait_timeout_selftest(_stream(stream)))
