"""Helpers shared by the GPU tests: move oracle-made parameters and records into the library, and read
device results back. Data only ever flows oracle -> CUDA path, never the other way."""
import math

import numpy as np
import torch

from oracle import kvtc_oracle as O
from transform_coded_kv_02_b300 import kvtc, synth

DEV = "cuda"


def lib_params(sets):
    """sets: list of (TensorParams K, TensorParams V) from the oracle -> uploaded library table."""
    pk0, pv0 = sets[0]
    P = kvtc.kv_params_from_arrays(
        np.stack([s[0].T for s in sets]), np.stack([s[0].mu for s in sets]), np.stack([s[0].sigma for s in sets]),
        np.stack([s[0].widths for s in sets]), pk0.r_words,
        np.stack([s[1].T for s in sets]), np.stack([s[1].mu for s in sets]), np.stack([s[1].sigma for s in sets]),
        np.stack([s[1].widths for s in sets]), pv0.r_words)
    return P.upload()


def calibrate_oracle(L, bits_k, bits_v):
    return [O.calibrate(ck, cv, cq, bits_k, bits_v) for ck, cv, cq in zip(L.calib_k, L.calib_v, L.calib_q)]


def to_dev_storage(x):
    """Storage-typed numpy array (fp32 or bf16 bits) -> CUDA tensor (float32 or bfloat16)."""
    if x.dtype == np.uint16:
        return torch.from_numpy(x.view(np.int16).copy()).to(DEV).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(x)).to(DEV)


def u32(t):
    return t.cpu().numpy().view(np.uint32)


def oracle_records(x, p):
    """x: [n, d] float64 raw vectors -> oracle records [n, R]."""
    return O.encode(x, p)


def set_index(b, h, Hkv, per_seq):
    return b * Hkv + h if per_seq else h


def value_cache_shape(B, Hkv, T_cap, r_words):
    """Value cache: two-token records of 2 R words, [B, Hkv, T_cap / 2, 2 R]."""
    return (B, Hkv, T_cap // 2, 2 * r_words)


def oracle_cache(k, v, sets, per_seq, T_cap=None):
    """Oracle-encoded records for k, v [B, Hkv, T, d] (float64) -> numpy uint32 key cache [B, Hkv, T_cap, R]
    and value cache [B, Hkv, T_cap / 2, 2 R] (T_cap even)."""
    B, Hkv, T, d = k.shape
    T_cap = T_cap or (T + T % 2)
    Rk, Rv = sets[0][0].r_words, sets[0][1].r_words
    rk = np.zeros((B, Hkv, T_cap, Rk), np.uint32)
    rv = np.zeros(value_cache_shape(B, Hkv, T_cap, Rv), np.uint32)
    for b in range(B):
        for h in range(Hkv):
            pk, pv = sets[set_index(b, h, Hkv, per_seq)]
            rk[b, h, :T] = O.encode(k[b, h], pk)
            rv[b, h, :(T + 1) // 2] = O.encode(v[b, h], pv)
    return rk, rv


def dev_u32(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int32)).to(DEV)


def run_decode(P, rk, rv, q_bits, seq_lens, Hq, per_seq, scale=None, T_cap=None):
    """rk: numpy uint32 [B, Hkv, T_cap, R]; rv: [B, Hkv, T_cap / 2, 2 R]; q_bits: bf16 bits [B, Hq, d];
    returns fp32 [B, Hq, d]."""
    B, Hkv, Tc, _ = rk.shape
    d = 128
    scale = scale if scale is not None else 1.0 / math.sqrt(d)
    tk, tv = dev_u32(rk), dev_u32(rv)
    cache = kvtc.make_cache(tk, tv, B, Hkv, Tc, per_seq)
    q = to_dev_storage(q_bits)
    sl = torch.tensor(seq_lens, dtype=torch.int32, device=DEV)
    out = torch.full((B, Hq, d), float("nan"), dtype=torch.float32, device=DEV)
    wsb = kvtc.kv_decode_workspace_bytes(P, B, Hkv, Hq, Tc)
    ws = torch.zeros(wsb, dtype=torch.uint8, device=DEV)  # zero-filled before first use (arrival counters)
    kvtc.kv_attend_decode(P, cache, q, B, Hq, sl, scale, out, ws)
    assert kvtc.kv_check_status() == kvtc.KV_OK, kvtc.kv_last_error()
    return out.cpu().numpy().astype(np.float64)


def oracle_decode(rk, rv, q_bits, seq_lens, sets, Hq, per_seq, scale=None):
    B, Hkv = rk.shape[:2]
    g = Hq // Hkv
    d = 128
    scale = scale if scale is not None else 1.0 / math.sqrt(d)
    q = synth.as_float(q_bits)
    out = np.zeros((B, Hq, d))
    for b in range(B):
        for h in range(Hkv):
            pk, pv = sets[set_index(b, h, Hkv, per_seq)]
            out[b, h * g:(h + 1) * g] = O.attend_decode(q[b, h * g:(h + 1) * g], rk[b, h], rv[b, h], pk, pv,
                                                        int(seq_lens[b]), scale)
    return out


def rel_l2_rows(a, b):
    """Relative L2 error of each (batch, head) output row."""
    num = np.linalg.norm((a - b).reshape(-1, a.shape[-1]), axis=1)
    den = np.linalg.norm(b.reshape(-1, b.shape[-1]), axis=1)
    return num / np.maximum(den, 1e-30)


def code_diff(rec_a, rec_b, p, n=None):
    """Compare two record sets: (fraction of tokens whose z or s differ, max |dz| and |ds| in fp16 ulps,
    fraction of code entries that differ, max |code difference|, fraction of all record entries - z, s and
    the codes of the nonzero-width channels - that differ)."""
    za, sa, ca = O.unpack(rec_a, p)
    zb, sb, cb = O.unpack(rec_b, p)
    if n is not None:
        za, sa, ca, zb, sb, cb = za[:n], sa[:n], ca[:n], zb[:n], sb[:n], cb[:n]
    return token_diff((za, sa, ca), (zb, sb, cb), p)


def token_diff(a, b, p):
    """code_diff on per-token unpacked records (z, s, codes) as O.unpack returns them."""
    za, sa, ca = a
    zb, sb, cb = b
    zi = lambda h: h.view(np.uint16).astype(np.int64)
    dz = np.abs(zi(za) - zi(zb))
    ds = np.abs(zi(sa) - zi(sb))
    nz = p.widths > 0
    dc = np.abs(ca[:, nz] - cb[:, nz])
    n_entries = dc.size + 2 * dz.size
    entry_frac = float((np.count_nonzero(dc) + np.count_nonzero(dz) + np.count_nonzero(ds)) / max(n_entries, 1))
    return (float(np.mean((dz > 0) | (ds > 0))), int(dz.max(initial=0)), int(ds.max(initial=0)),
            float(np.mean(dc > 0)), int(dc.max(initial=0)), entry_frac)


def tokens_of(rec, p, start, n):
    """Per-token (z, s, codes) of tokens start .. start + n - 1 of a cache row (keys [T_cap, R], values
    [T_cap / 2, 2 R]); the value record of an odd start is shared with the token before it."""
    z, s, c = O.unpack(rec, p)
    return z[start:start + n], s[start:start + n], c[start:start + n]
