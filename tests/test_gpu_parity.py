"""Parity of the CUDA path (through the C-ABI) with the CPU oracle on the same seeded inputs.

Bars: quantise+pack and unpack bit-exact given the same fp32 rotated input; end-to-end codes differ by at most
1 LSB on at most 1e-4 of entries (rounding ties of the rotation); decode within 2e-3 relative L2 of the oracle
run on the same records."""
import dataclasses
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

from oracle import kvtc_oracle as O
from transform_coded_kv_02_b300 import kvtc, synth

import gpu_helpers as G

pytestmark = pytest.mark.gpu
DEC_TOL = 2e-3


@pytest.fixture(scope="module")
def tiny():
    w = synth.WORKLOADS["tiny"]
    L = synth.make_layer(w, steps=2)
    sets = G.calibrate_oracle(L, 2.75, 2.75)
    return w, L, sets, G.lib_params(sets)


def _special_rows(p, rng, n=64):
    """Rotated fp32 rows with the codec's corner cases: constant rows (s = 0), saturating magnitudes,
    tiny magnitudes (subnormal fp16 z/s), negative zero, values on a coarse grid (exact bin edges)."""
    d = p.d
    mu, sg = p.mu.astype(np.float64), p.sigma.astype(np.float64)
    rows = [np.full(d, mu[0]), mu.copy(), mu + 1e6 * sg, mu - 3e5 * sg * np.sign(np.arange(d) - 60.5),
            mu + 1e-7 * sg * rng.normal(size=d), mu + 1e-9 * sg * rng.normal(size=d), -mu * 0.0]
    grid = mu + sg * (np.round(rng.normal(size=(n, d)) * 4) / 4)
    rows = np.vstack([np.array(rows), grid, mu + sg * rng.normal(size=(n, d)) * 3])
    return rows.astype(np.float32)


def _near_tie_rows(p, rng, n_rows=24):
    """Rotated fp32 rows whose normalised coefficients sit on a quantiser bin edge or a few fp32 ulps from one.
    In each row every coded channel other than the row's extremes (which fix z and s) is aimed at
    y' = z + s k 2^-b_j for a random interior edge k, then moved ulp by ulp (17 candidates) to the y whose
    quotient (y' - z) / s 2^b_j lands closest to k from the side the row asks for: just below, as close as fp32
    gets, or just above."""
    nz = np.nonzero(p.widths > 0)[0]
    mu, inv, sg = p.mu, p.inv_sigma, p.sigma
    rows = []
    for r in range(n_rows):
        y = (mu + sg * rng.normal(size=p.d).astype(np.float32) * 2).astype(np.float32)
        yp = (y[nz] - mu[nz]) * inv[nz]
        jmin, jmax = nz[np.argmin(yp)], nz[np.argmax(yp)]
        z = np.float64(O.half_rn_sat(yp.min()))
        s = np.float64(O.half_rn_sat(np.float32(yp.max() - np.float32(z))))
        side = r % 3
        for j in nz:
            if j in (jmin, jmax):
                continue
            b = int(p.widths[j])
            k = int(rng.integers(1, 2 ** b))
            y0 = np.float32((z + s * k / 2.0 ** b) / np.float64(inv[j]) + np.float64(mu[j]))
            bits0 = np.array([y0], np.float32).view(np.int32)[0]
            best, bestd = y0, None
            for step in range(-8, 9):
                c = np.array([bits0 + step], np.int32).view(np.float32)[0]
                d = (np.float64((c - mu[j]) * inv[j]) - z) / s * 2.0 ** b - k
                ok, key = ((d < 0, -d), (True, abs(d)), (d >= 0, d))[side]
                if ok and (bestd is None or key < bestd):
                    best, bestd = c, key
            y[j] = best
        rows.append(y)
    return np.array(rows, np.float32)


def _reciprocal_only_codes(y, p):
    """Codes of the coded channels as the reciprocal quotient alone would give them (u = (y' - z) (RN(1/s) 2^b),
    clamped to [1/2, 2^b - 1/2], floored), i.e. without the tensor-core epilogue's exact redo of near-ties."""
    nz = p.widths > 0
    yp = (y[:, nz] - p.mu[nz]) * p.inv_sigma[nz]
    z = O.half_rn_sat(yp.min(1)).astype(np.float32)
    s = O.half_rn_sat(yp.max(1) - z).astype(np.float32)
    tb = np.ldexp(np.ones(int(nz.sum()), np.float32), p.widths[nz].astype(np.int32))
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        u = (yp - z[:, None]) * ((np.float32(1) / s)[:, None] * tb[None, :])
        c = np.floor(np.minimum(np.maximum(u, np.float32(0.5)), tb - np.float32(0.5)))
    c[s == 0] = 0
    return c.astype(np.int64)


@pytest.mark.parametrize("variant", [0, 1, 2])
@pytest.mark.parametrize("bits", [2.75, 1.33, 4.0, 8.0])
def test_quantize_pack_bitexact(tiny, variant, bits):
    """The three device quantisers (variant 0: warp per token, CUDA-core encode; 1: thread per token; 2: the
    tensor-core encode's epilogue, run on coefficients stored into tensor memory) against the oracle's
    quantiser and packer on the same fp32 rotated rows: bit-exact records. Rows: the tiny layer's rotated tokens,
    the codec's corner cases (s = 0, saturation, subnormal z and s, -0, exact bin edges on a coarse grid) and
    rows of near-ties; 1024 + 159 rows, so variant 2 also ends on a ragged tile."""
    w, L, _, _ = tiny
    sets = G.calibrate_oracle(L, bits, bits)
    P = G.lib_params(sets)
    rng = np.random.default_rng(100)
    for t, p in ((0, sets[0][0]), (1, sets[0][1])):
        x = synth.as_float(L.k[0, 0] if t == 0 else L.v[0, 0])
        y = np.vstack([O.rotate(x, p), _special_rows(p, rng), _near_tie_rows(p, rng)])
        ref = O.pack(*O.quantize(y, p), p)
        if variant == 2:  # the near-tie rows do reach the exact redo: the reciprocal alone differs somewhere
            assert np.count_nonzero(_reciprocal_only_codes(y, p) != O.quantize(y, p)[2][:, p.widths > 0]) > 0
        yd = torch.from_numpy(y).cuda()
        rec = torch.zeros(ref.shape, dtype=torch.int32, device="cuda")
        kvtc.kv_debug_quantize_pack(P, 0, t, yd, y.shape[0], rec, variant)
        assert kvtc.kv_check_status() == kvtc.KV_OK
        got = G.u32(rec)
        bad = np.argwhere(got != ref)
        assert bad.size == 0, (t, bad[:5], got[bad[0][0]], ref[bad[0][0]])


@pytest.mark.parametrize("bits", [2.75, 1.33, 3.0, 8.0])
def test_unpack_bitexact(tiny, bits):
    w, L, _, _ = tiny
    sets = G.calibrate_oracle(L, bits, bits)
    P = G.lib_params(sets)
    for t, p in ((0, sets[0][0]), (1, sets[0][1])):
        n = 333  # odd: the last value record holds one token
        x = synth.as_float(L.k[0, 0] if t == 0 else L.v[0, 0])[:n]
        rec = O.encode(x, p)
        codes = O.unpack(rec, p)[2][:n]
        out = torch.zeros((n, 128), dtype=torch.int16, device="cuda")
        kvtc.kv_debug_unpack(P, 0, t, G.dev_u32(rec), n, out)
        assert kvtc.kv_check_status() == kvtc.KV_OK
        got = out.cpu().numpy().view(np.uint16).astype(np.int64)
        assert np.array_equal(got, codes)


def _encode_gpu(P, k_st, v_st, per_seq, T_cap=None, dst0=0):
    B, Hkv, T, d = k_st.shape
    T_cap = T_cap or ((T + 15) // 16 * 16)
    Rk, Rv = P.record_words(0), P.record_words(1)
    rk = torch.zeros((B, Hkv, T_cap, Rk), dtype=torch.int32, device="cuda")
    rv = torch.zeros(G.value_cache_shape(B, Hkv, T_cap, Rv), dtype=torch.int32, device="cuda")
    cache = kvtc.make_cache(rk, rv, B, Hkv, T_cap, per_seq)
    dt = kvtc.KV_DTYPE_BF16 if k_st.dtype == np.uint16 else kvtc.KV_DTYPE_F32
    pos = torch.full((B,), dst0, dtype=torch.int64, device="cuda")
    kvtc.kv_encode(P, cache, G.to_dev_storage(k_st), G.to_dev_storage(v_st), dt, B, T, pos)
    assert kvtc.kv_check_status() == kvtc.KV_OK, kvtc.kv_last_error()
    return G.u32(rk), G.u32(rv)


def _check_end_to_end(rk_gpu, rv_gpu, k, v, sets, per_seq):
    """End-to-end encode against the oracle: every record entry (fp16 z, fp16 s, and the code of each
    nonzero-width channel) within 1 LSB, and at most 1e-4 of all entries different. The rotation's fp32
    rounding on the device differs from the oracle's single rounding of an fp64 product, so a value that
    lands within an ulp of a quantiser bin edge or an fp16 rounding boundary can move by one step."""
    B, Hkv, T, _ = k.shape
    tok_frac, code_frac, entry_frac, max_dc, max_dz = 0.0, 0.0, 0.0, 0, 0
    n = 0
    for b in range(B):
        for h in range(Hkv):
            pk, pv = sets[G.set_index(b, h, Hkv, per_seq)]
            for rec, x, p in ((rk_gpu[b, h, :T], k[b, h], pk), (rv_gpu[b, h, :(T + 1) // 2], v[b, h], pv)):
                ref = O.encode(x, p)
                tf, dz, ds, cf, dc, ef = G.code_diff(rec, ref, p, T)
                tok_frac += tf
                code_frac += cf
                entry_frac += ef
                max_dc = max(max_dc, dc)
                max_dz = max(max_dz, dz, ds)
                n += 1
    tok_frac /= n
    code_frac /= n
    entry_frac /= n
    assert max_dc <= 1 and max_dz <= 1, (max_dc, max_dz)
    assert entry_frac <= 1e-4, (entry_frac, code_frac, tok_frac)
    return entry_frac, code_frac, tok_frac


def test_encode_end_to_end_tiny_fp32(tiny):
    w, L, sets, P = tiny
    rk, rv = _encode_gpu(P, L.k, L.v, False)
    print("entry mismatch fraction %.2e, code mismatch fraction %.2e, token z/s mismatch fraction %.2e" %
          _check_end_to_end(rk, rv, synth.as_float(L.k), synth.as_float(L.v), sets, False))


def test_encode_end_to_end_bf16_per_sequence():
    w = synth.WORKLOADS["qwen_batched_8k"]
    L = synth.make_layer(w, T=1024, B=2, steps=1)
    for bits in w.bits:
        sets = G.calibrate_oracle(L, bits, bits)
        P = G.lib_params(sets)
        rk, rv = _encode_gpu(P, L.k, L.v, True)
        _check_end_to_end(rk, rv, synth.as_float(L.k), synth.as_float(L.v), sets, True)


@pytest.fixture(scope="module")
def llama_300():
    """Llama-shaped layer (8 KV heads, bf16, RoPE on keys, one parameter set per head) with 300 new tokens:
    two full 128-token tiles and a ragged one per head."""
    w = synth.WORKLOADS["llama_decode_32k"]
    L = synth.make_layer(w, T=300, steps=1)
    sets = G.calibrate_oracle(L, 2.75, 2.75)
    return w, L, sets, G.lib_params(sets)


def _check_tokens(rk, rv, k, v, sets, per_seq, dst0, T, frac_bar=1e-4):
    """Every token's record entries at cache positions dst0 .. dst0 + T - 1 against the oracle encode of the
    same vectors: each entry within 1 LSB, at most frac_bar of all the entries checked different, and nothing
    written outside those positions."""
    B, Hkv = k.shape[:2]
    n_diff, n_all = 0.0, 0
    for b in range(B):
        for h in range(Hkv):
            pk, pv = sets[G.set_index(b, h, Hkv, per_seq)]
            for rec, x, p in ((rk[b, h], k[b, h], pk), (rv[b, h], v[b, h], pv)):
                got = G.tokens_of(rec, p, dst0, T)
                ref = G.tokens_of(O.encode(x, p), p, 0, T)
                tf, dz, ds, cf, dc, ef = G.token_diff(got, ref, p)
                assert dc <= 1 and dz <= 1 and ds <= 1, (b, h, dz, ds, dc)
                n = T * (int(np.count_nonzero(p.widths)) + 2)
                n_diff += ef * n
                n_all += n
                z, s, c = O.unpack(rec, p)
                outside = np.r_[0:dst0, dst0 + T:len(z)]
                assert not np.any(z.view(np.uint16)[outside]) and not np.any(s.view(np.uint16)[outside])
                assert not np.any(c[outside])
    frac = n_diff / n_all
    assert frac <= frac_bar, (frac, round(n_diff), n_all)
    return frac


@pytest.mark.parametrize("path", [1, 2])
@pytest.mark.parametrize("dst0", [0, 5])
def test_encode_paths_bf16_llama_shape(llama_300, path, dst0):
    """The CUDA-core path and the tensor-core path against the oracle on 8 bf16 heads with a ragged last tile;
    an odd write offset makes value records straddle tile edges and share a record with an unwritten token."""
    w, L, sets, P = llama_300
    kvtc.kv_debug_set_encode_path(path)
    try:
        rk, rv = _encode_gpu(P, L.k, L.v, False, T_cap=320, dst0=dst0)
    finally:
        kvtc.kv_debug_set_encode_path(0)
    _check_tokens(rk, rv, synth.as_float(L.k), synth.as_float(L.v), sets, False, dst0, L.k.shape[2])


@pytest.mark.parametrize("bits", [1.33, 4.0, 8.0])
def test_encode_tensor_core_budgets_per_sequence(bits):
    """Tensor-core encode at 5, 16 and 32 record words (four epilogue groups at 5 and 16 words; at 32 the record
    staging only fits three), one parameter set per (sequence, head).

    The 1e-4 mismatch bar belongs to the workloads' budgets (at most 4 bits per element). A code flips when the
    fp32 rotation's rounding error carries a value across a bin edge, so the flip rate scales with 1 / bin
    width: at 8 bits per element the channels get 7-8 bits instead of 3-4, bins 16 times narrower than at
    4 bits, and the bar scales to 16e-4. Every entry must still be within 1 LSB."""
    w = synth.WORKLOADS["qwen_batched_8k"]
    L = synth.make_layer(w, T=200, B=2, steps=1)
    sets = G.calibrate_oracle(L, bits, bits)
    P = G.lib_params(sets)
    kvtc.kv_debug_set_encode_path(2)
    try:
        rk, rv = _encode_gpu(P, L.k, L.v, True, T_cap=208, dst0=3)
    finally:
        kvtc.kv_debug_set_encode_path(0)
    _check_tokens(rk, rv, synth.as_float(L.k), synth.as_float(L.v), sets, True, 3, 200,
                  frac_bar=1.6e-3 if bits > 4 else 1e-4)


def test_encode_tensor_core_rejects_fp32(tiny):
    w, L, sets, P = tiny
    kvtc.kv_debug_set_encode_path(2)
    try:
        k, v = np.ascontiguousarray(L.k[:, :, :128]), np.ascontiguousarray(L.v[:, :, :128])
        rk = torch.zeros((1, 1, 128, P.record_words(0)), dtype=torch.int32, device="cuda")
        rv = torch.zeros(G.value_cache_shape(1, 1, 128, P.record_words(1)), dtype=torch.int32, device="cuda")
        cache = kvtc.make_cache(rk, rv, 1, 1, 128, False)
        pos = torch.zeros((1,), dtype=torch.int64, device="cuda")
        with pytest.raises(kvtc.KvError) as e:
            kvtc.kv_encode(P, cache, G.to_dev_storage(k), G.to_dev_storage(v), kvtc.KV_DTYPE_F32, 1, 128, pos)
        assert e.value.status == kvtc.KV_ERR_UNSUPPORTED
    finally:
        kvtc.kv_debug_set_encode_path(0)


def test_encode_full_size_llama_32k_sampled():
    """Prefill of the 32K-token Llama-shaped layer through kv_encode in its default configuration (the
    tensor-core path): 1024 sampled token pairs per head against the oracle encode of the same vectors."""
    w = synth.WORKLOADS["llama_decode_32k"]
    L = synth.make_layer(w, steps=1)
    sets = G.calibrate_oracle(L, 2.75, 2.75)
    P = G.lib_params(sets)
    T = w.T
    rk, rv = _encode_gpu(P, L.k, L.v, False, T_cap=T + 512)
    rng = np.random.default_rng(7)
    n_diff, n_all = 0.0, 0
    for h in range(w.Hkv):
        pk, pv = sets[h]
        pairs = np.sort(rng.choice(T // 2, 1024, replace=False))
        toks = np.stack([2 * pairs, 2 * pairs + 1], 1).reshape(-1)
        kx, vx = synth.as_float(L.k[0, h, toks]), synth.as_float(L.v[0, h, toks])
        ga = O.unpack(rk[0, h, toks], pk)
        gv = O.unpack(rv[0, h, pairs], pv)
        for got, ref, p in ((ga, O.unpack(O.encode(kx, pk), pk), pk), (gv, O.unpack(O.encode(vx, pv), pv), pv)):
            tf, dz, ds, cf, dc, ef = G.token_diff(got, ref, p)
            assert dc <= 1 and dz <= 1 and ds <= 1, (h, dz, ds, dc)
            n = len(toks) * (int(np.count_nonzero(p.widths)) + 2)
            n_diff += ef * n
            n_all += n
    assert n_diff / n_all <= 1e-4, (n_diff / n_all, round(n_diff), n_all)


def test_append_matches_prefill(tiny):
    w, L, sets, P = tiny
    T = 200
    k, v = L.k[:, :, :T], L.v[:, :, :T]
    rk_all, rv_all = _encode_gpu(P, k, v, False, T_cap=256)
    rk = torch.zeros((1, 1, 256, P.record_words(0)), dtype=torch.int32, device="cuda")
    rv = torch.zeros(G.value_cache_shape(1, 1, 256, P.record_words(1)), dtype=torch.int32, device="cuda")
    cache = kvtc.make_cache(rk, rv, 1, 1, 256, False)
    kd, vd = G.to_dev_storage(np.ascontiguousarray(k)), G.to_dev_storage(np.ascontiguousarray(v))
    for i in range(T):
        pos = torch.tensor([i], dtype=torch.int64, device="cuda")
        kvtc.kv_encode(P, cache, kd[:, :, i:i + 1].contiguous(), vd[:, :, i:i + 1].contiguous(),
                       kvtc.KV_DTYPE_F32, 1, 1, pos)
    assert kvtc.kv_check_status() == kvtc.KV_OK
    assert np.array_equal(G.u32(rk), rk_all) and np.array_equal(G.u32(rv), rv_all)


def _value_token_raw(rec, t):
    """Raw bits of token t in a value cache row [T_cap / 2, 2 R]: its z/s word (word t & 1 of its record) and
    its 16-bit half (t & 1) of every code word."""
    r = rec[t >> 1]
    return np.concatenate([[r[t & 1]], (r[2:].astype(np.uint32) >> (16 * (t & 1))) & 0xFFFF])


@pytest.mark.parametrize("wl,bits", [("llama_decode_32k", 2.75), ("qwen_batched_8k", 3.0)])
def test_append_bf16_one_token_per_call_matches_oracle(wl, bits):
    """The bf16 append kernel (t_new = 1 per call: the encode of every decode step) against the oracle. Two
    sequences, 70 tokens each, appended one call at a time into a cache pre-filled with the oracle's records of
    other tokens; sequence 0 starts at an even position and sequence 1 at an odd one, so the first and the last
    value records are shared with a background token. Every appended token's record entries are within 1 LSB of
    the oracle's with at most 1e-4 of them different; every other token of the cache, including the other half
    of each shared value record, keeps its bits."""
    w = synth.WORKLOADS[wl]
    n_bg, n_app, T_cap, starts = 96, 70, 96, (4, 9)
    L = synth.make_layer(w, T=n_bg + n_app, B=2, steps=1)
    sets = G.calibrate_oracle(L, bits, bits)
    P = G.lib_params(sets)
    per_seq = L.per_seq_params
    kf, vf = synth.as_float(L.k), synth.as_float(L.v)
    bg_k, bg_v = G.oracle_cache(kf[:, :, :n_bg], vf[:, :, :n_bg], sets, per_seq, T_cap)
    rk, rv = G.dev_u32(bg_k), G.dev_u32(bg_v)
    cache = kvtc.make_cache(rk, rv, 2, w.Hkv, T_cap, per_seq)
    kn = G.to_dev_storage(np.ascontiguousarray(L.k[:, :, n_bg:]))
    vn = G.to_dev_storage(np.ascontiguousarray(L.v[:, :, n_bg:]))
    for i in range(n_app):
        pos = torch.tensor([starts[0] + i, starts[1] + i], dtype=torch.int64, device="cuda")
        kvtc.kv_encode(P, cache, kn[:, :, i:i + 1].contiguous(), vn[:, :, i:i + 1].contiguous(), kvtc.KV_DTYPE_BF16,
                       2, 1, pos)
    assert kvtc.kv_check_status() == kvtc.KV_OK, kvtc.kv_last_error()
    got_k, got_v = G.u32(rk), G.u32(rv)
    n_diff, n_all = 0.0, 0
    for b in range(2):
        s0 = starts[b]
        keep = [t for t in range(T_cap) if not s0 <= t < s0 + n_app]
        for h in range(w.Hkv):
            pk, pv = sets[G.set_index(b, h, w.Hkv, per_seq)]
            for got, bg, x, p in ((got_k[b, h], bg_k[b, h], kf[b, h, n_bg:], pk),
                                  (got_v[b, h], bg_v[b, h], vf[b, h, n_bg:], pv)):
                z, s, c = O.unpack(got, p)
                ref = O.unpack(O.encode(x, p), p)
                tf, dz, ds, cf, dc, ef = G.token_diff((z[s0:s0 + n_app], s[s0:s0 + n_app], c[s0:s0 + n_app]),
                                                      tuple(a[:n_app] for a in ref), p)
                assert dc <= 1 and dz <= 1 and ds <= 1, (b, h, p.pairing, dz, ds, dc)
                n = n_app * (int(np.count_nonzero(p.widths)) + 2)
                n_diff += ef * n
                n_all += n
                raw = (lambda r, t: r[t]) if p.pairing == "channels" else _value_token_raw
                for t in keep:
                    assert np.array_equal(raw(got, t), raw(bg, t)), (b, h, p.pairing, t)
    assert n_diff / n_all <= 1e-4, (n_diff / n_all, round(n_diff), n_all)


def test_encode_out_of_range_position_is_reported(tiny):
    w, L, sets, P = tiny
    k, v = np.ascontiguousarray(L.k[:, :, :4]), np.ascontiguousarray(L.v[:, :, :4])
    rk = torch.zeros((1, 1, 64, P.record_words(0)), dtype=torch.int32, device="cuda")
    rv = torch.zeros(G.value_cache_shape(1, 1, 64, P.record_words(1)), dtype=torch.int32, device="cuda")
    cache = kvtc.make_cache(rk, rv, 1, 1, 64, False)
    pos = torch.tensor([62], dtype=torch.int64, device="cuda")  # tokens 2, 3 fall past T_cap
    kvtc.kv_encode(P, cache, G.to_dev_storage(k), G.to_dev_storage(v), kvtc.KV_DTYPE_F32, 1, 4, pos)
    assert kvtc.kv_check_status() == kvtc.KV_ERR_DEVICE
    ref = O.encode(synth.as_float(L.k[0, 0, :2]), sets[0][0])
    tok, dz, ds, cf, dc, ef = G.code_diff(G.u32(rk)[0, 0, 62:64], ref, sets[0][0])
    assert dc <= 1 and dz <= 1 and ds <= 1
    assert kvtc.kv_check_status() == kvtc.KV_OK  # cleared


def _decode_case(L, sets, P, Hq, per_seq, seq_lens, T_cap, scale=None):
    k, v = synth.as_float(L.k), synth.as_float(L.v)
    rk, rv = G.oracle_cache(k, v, sets, per_seq, T_cap)
    q = L.q[0]
    got = G.run_decode(P, rk, rv, q, seq_lens, Hq, per_seq, scale)
    ref = G.oracle_decode(rk, rv, q, seq_lens, sets, Hq, per_seq, scale)
    return G.rel_l2_rows(got, ref)


def test_decode_tiny(tiny):
    w, L, sets, P = tiny
    err = _decode_case(L, sets, P, w.Hq, False, [w.T], 1024)
    assert err.max() <= DEC_TOL, err


@pytest.mark.parametrize("seq_len", [1, 2, 3, 15, 16, 17, 31, 33, 63, 64, 65, 100, 127, 129, 1000])
def test_decode_ragged_lengths(tiny, seq_len):
    w, L, sets, P = tiny
    err = _decode_case(L, sets, P, w.Hq, False, [seq_len], 1024)
    assert err.max() <= DEC_TOL, (seq_len, err)


def test_decode_split_count_invariance(tiny):
    """Different cache capacities give different split plans over the same 1000 tokens. The results differ
    only by rounding: fp32 merge order, and the fp16 hi/lo split of p*s taken against each split's running
    maximum (about 1e-5 relative); a merge mistake would be of order one."""
    w, L, sets, P = tiny
    k, v = synth.as_float(L.k), synth.as_float(L.v)
    outs = []
    for T_cap in (1024, 4096, 65536):
        rk, rv = G.oracle_cache(k, v, sets, False, T_cap)
        outs.append(G.run_decode(P, rk, rv, L.q[0], [1000], w.Hq, False))
    for o in outs[1:]:
        assert G.rel_l2_rows(o, outs[0]).max() <= 1e-4


@pytest.mark.parametrize("bits", [2.0, 3.0, 4.0])
def test_decode_qwen_shape_per_sequence(bits):
    w = synth.WORKLOADS["qwen_batched_8k"]
    L = synth.make_layer(w, T=512, B=2, steps=1)
    sets = G.calibrate_oracle(L, bits, bits)
    P = G.lib_params(sets)
    err = _decode_case(L, sets, P, w.Hq, True, [512, 300], 512)
    assert err.max() <= DEC_TOL, err


def test_decode_high_compression_llama_shape():
    w = synth.WORKLOADS["llama_long_128k"]
    L = synth.make_layer(w, T=2048, steps=1)
    sets = G.calibrate_oracle(L, 1.33, 1.33)
    P = G.lib_params(sets)
    err = _decode_case(L, sets, P, w.Hq, False, [2048], 2048)
    assert err.max() <= DEC_TOL, err


def test_decode_other_softmax_scale(tiny):
    w, L, sets, P = tiny
    err = _decode_case(L, sets, P, w.Hq, False, [777], 1024, scale=0.3)
    assert err.max() <= DEC_TOL, err


def test_decode_bf16_comparator_matches_exact_attention():
    w = synth.WORKLOADS["qwen_batched_8k"]
    L = synth.make_layer(w, T=700, B=2, steps=1)
    B, Hkv, T, d = L.k.shape
    T_cap = 704
    kp = np.zeros((B, Hkv, T_cap, d), np.uint16)
    vp = np.zeros((B, Hkv, T_cap, d), np.uint16)
    kp[:, :, :T] = L.k
    vp[:, :, :T] = L.v
    seq = [700, 333]
    q = L.q[0]
    kd, vd, qd = G.to_dev_storage(kp), G.to_dev_storage(vp), G.to_dev_storage(q)
    sl = torch.tensor(seq, dtype=torch.int32, device="cuda")
    out = torch.empty((B, w.Hq, d), dtype=torch.float32, device="cuda")
    ws = torch.zeros(kvtc.kv_decode_bf16_workspace_bytes(B, Hkv, w.Hq, T_cap), dtype=torch.uint8, device="cuda")
    scale = 1 / math.sqrt(d)
    kvtc.kv_attend_decode_bf16(kd, vd, B, Hkv, w.Hq, T_cap, qd, sl, scale, out, ws)
    assert kvtc.kv_check_status() == kvtc.KV_OK
    got = out.cpu().numpy().astype(np.float64)
    kf, vf, qf = synth.as_float(kp), synth.as_float(vp), synth.as_float(q)
    g = w.g
    ref = np.zeros_like(got)
    for b in range(B):
        for h in range(Hkv):
            ref[b, h * g:(h + 1) * g] = O.attention(qf[b, h * g:(h + 1) * g], kf[b, h, :seq[b]], vf[b, h, :seq[b]],
                                                    scale)
    err = G.rel_l2_rows(got, ref)
    assert err.max() <= 1e-4, err


@pytest.mark.parametrize("seq_len", [1, 63, 1000, 2048])
def test_decode_llama_shape_all_key_blocks(seq_len):
    """Llama-shaped keys fill all eight 16-channel blocks (the decode's eight-block kernel); ragged lengths exercise
    its partial last stage."""
    w = synth.WORKLOADS["llama_decode_32k"]
    L = synth.make_layer(w, T=2048, steps=1)
    sets = G.calibrate_oracle(L, 2.75, 2.75)
    assert min(int(np.max(np.nonzero(s[0].widths)[0])) + 1 for s in sets) > 96
    P = G.lib_params(sets)
    err = _decode_case(L, sets, P, w.Hq, False, [seq_len], 2048)
    assert err.max() <= DEC_TOL, (seq_len, err)


@pytest.mark.parametrize("wl,bits", [("llama_decode_32k", 8.0), ("qwen_batched_8k", 6.0)])
def test_decode_runtime_record_length(wl, bits):
    """Record lengths without a compile-time kernel (32 words at 8 bits per element, 24 at 6) run the decode with
    run-time record strides: one column block on the Llama shape, two column blocks
    on the Qwen shape, ragged lengths. The wide codes also give the smallest q' entries (sigma_j 2^-b_j near
    1e-6), which the per-head power-of-two scaling of q' keeps out of the fp16 subnormal range."""
    w = synth.WORKLOADS[wl]
    L = synth.make_layer(w, T=1000, B=min(w.B, 2), steps=1)
    sets = G.calibrate_oracle(L, bits, bits)
    assert sets[0][0].r_words not in (5, 8, 11, 12, 16)
    P = G.lib_params(sets)
    seq = [1000, 777][:L.k.shape[0]]
    err = _decode_case(L, sets, P, w.Hq, L.per_seq_params, seq, 1024)
    print("decode rel-L2 max %.2e" % err.max())
    assert err.max() <= DEC_TOL, err


def test_encode_zero_tokens_is_a_no_op(tiny):
    """t_new = 0 returns at once, before any pointer is looked at, and writes nothing."""
    w, L, sets, P = tiny
    rk = torch.full((1, 1, 64, P.record_words(0)), 7, dtype=torch.int32, device="cuda")
    rv = torch.full(G.value_cache_shape(1, 1, 64, P.record_words(1)), 7, dtype=torch.int32, device="cuda")
    cache = kvtc.make_cache(rk, rv, 1, 1, 64, False)
    kvtc.kv_encode(P, cache, None, None, kvtc.KV_DTYPE_F32, 1, 0, None)
    assert kvtc.kv_check_status() == kvtc.KV_OK
    assert bool(torch.all(rk == 7)) and bool(torch.all(rv == 7))


def test_decode_empty_sequence_gives_zeros():
    """A batch whose first sequence is empty (seq_len 0): its rows are zeros, as the header states; the other
    sequence's rows match the oracle."""
    w = synth.WORKLOADS["qwen_batched_8k"]
    L = synth.make_layer(w, T=300, B=2, steps=1)
    sets = G.calibrate_oracle(L, 3.0, 3.0)
    P = G.lib_params(sets)
    rk, rv = G.oracle_cache(synth.as_float(L.k), synth.as_float(L.v), sets, True, 320)
    got = G.run_decode(P, rk, rv, L.q[0], [0, 300], w.Hq, True)
    assert np.all(got[0] == 0)
    ref = G.oracle_decode(rk[1:2], rv[1:2], L.q[0][1:2], [300], sets[w.Hkv:], w.Hq, True)
    assert G.rel_l2_rows(got[1:2], ref).max() <= DEC_TOL


def test_all_channels_at_zero_width():
    """The degenerate budget: 1-word records (0.25 bits per element) leave no code bits, so every channel has
    width 0. The tensor-core encode writes all-zero records like the oracle, and the decode returns the mean
    value T_V^T mu_V for every head (every key reconstructs to the same mean, so the softmax is uniform)."""
    w = synth.WORKLOADS["llama_decode_32k"]
    L = synth.make_layer(w, T=300, steps=1)
    sets = G.calibrate_oracle(L, 0.25, 0.25)
    assert all(s[0].r_words == 1 and not s[0].widths.any() and not s[1].widths.any() for s in sets)
    P = G.lib_params(sets)
    rk, rv = _encode_gpu(P, L.k, L.v, False, T_cap=320)
    assert not rk.any() and not rv.any()
    ork, orv = G.oracle_cache(synth.as_float(L.k), synth.as_float(L.v), sets, False, 320)
    got = G.run_decode(P, ork, orv, L.q[0], [300], w.Hq, False)
    ref = G.oracle_decode(ork, orv, L.q[0], [300], sets, w.Hq, False)
    assert G.rel_l2_rows(got, ref).max() <= DEC_TOL


def test_decode_largest_group():
    """g = 8 query heads per KV head, the library's largest group (two full column blocks)."""
    w = dataclasses.replace(synth.WORKLOADS["llama_decode_32k"], Hq=64)
    L = synth.make_layer(w, T=700, steps=1)
    sets = G.calibrate_oracle(L, 2.75, 2.75)
    P = G.lib_params(sets)
    err = _decode_case(L, sets, P, w.Hq, False, [700], 704)
    assert err.max() <= DEC_TOL, err


def test_joint_split_unequal_record_lengths():
    """The joint key/value split gives the Llama-shaped layer 14 key and 8 value words per token: the
    tensor-core encode and the decode with different record lengths for the two tensors, against the oracle."""
    w = synth.WORKLOADS["llama_decode_32k"]
    L = synth.make_layer(w, T=500, steps=1)
    sets = O.calibrate_joint(list(zip(L.calib_k, L.calib_v, L.calib_q)), 2.75, 2.75)
    assert (sets[0][0].r_words, sets[0][1].r_words) == (14, 8)
    P = G.lib_params(sets)
    rk, rv = _encode_gpu(P, L.k, L.v, False, T_cap=512)
    _check_tokens(rk, rv, synth.as_float(L.k), synth.as_float(L.v), sets, False, 0, 500)
    err = _decode_case(L, sets, P, w.Hq, False, [500], 512)
    assert err.max() <= DEC_TOL, err


def test_decode_full_size_llama_32k():
    """The 32K-token Llama-shaped layer (32 q / 8 KV heads, 2.75 bits) in the bench's launch configuration:
    every output row against the oracle on the same records."""
    w = synth.WORKLOADS["llama_decode_32k"]
    L = synth.make_layer(w, steps=1)
    sets = G.calibrate_oracle(L, 2.75, 2.75)
    P = G.lib_params(sets)
    T_cap = w.T + 512
    err = _decode_case(L, sets, P, w.Hq, False, [w.T], T_cap)
    assert err.max() <= DEC_TOL, err


def test_wait_timeout_is_reported_not_hung():
    kvtc.kv_debug_set_wait_limit_ns(1_000_000)
    try:
        kvtc.kv_debug_wait_timeout_selftest()
        assert kvtc.kv_check_status() == kvtc.KV_ERR_TIMEOUT
        assert kvtc.kv_check_status() == kvtc.KV_OK
    finally:
        kvtc.kv_debug_set_wait_limit_ns(2_000_000_000)


# ---- full sizes, at the cache capacity of bench.py's default run (8 warm-up + 256 timed steps, one appended
# token each), which fixes the decode's split plan ----
BENCH_APPENDED = 8 + 256


def _bench_T_cap(T):
    return (T + BENCH_APPENDED + 15) // 16 * 16


def _compare_records(got, ref, p, T):
    """Device records against the oracle's for the first T tokens of one cache row (keys [T_cap, R], values
    [T_cap / 2, 2 R]): identical words are equal records; records with any different word are unpacked and
    compared entry by entry. Returns (entries that differ, entries compared); asserts every entry within 1 LSB
    and nothing written past token T."""
    n_rec = (T + p.tokens_per_record - 1) // p.tokens_per_record
    assert not np.any(got[n_rec:]), "records written past the last token"
    if T % p.tokens_per_record:  # the unused token of the last value record stays zero
        z, s, c = O.unpack(got[n_rec - 1:n_rec], p)
        assert not (z.view(np.uint16)[1] or s.view(np.uint16)[1] or np.any(c[1])), "token T written"
    rows = np.nonzero(np.any(got[:n_rec] != ref[:n_rec], axis=1))[0]
    n_entries = T * (int(np.count_nonzero(p.widths)) + 2)
    if rows.size == 0:
        return 0, n_entries
    tf, dz, ds, cf, dc, ef = G.token_diff(O.unpack(got[rows], p), O.unpack(ref[rows], p), p)
    assert dc <= 1 and dz <= 1 and ds <= 1, (dz, ds, dc)
    n_rows_entries = rows.size * p.tokens_per_record * (int(np.count_nonzero(p.widths)) + 2)
    return ef * n_rows_entries, n_entries


def _full_size_case(w, L, bits):
    """kv_encode of the whole prefill (default path: tensor cores) against the oracle's records, every entry;
    then kv_attend_decode over the oracle's records against the oracle decode, every output row."""
    sets = G.calibrate_oracle(L, bits, bits)
    P = G.lib_params(sets)
    per_seq = L.per_seq_params
    B, Hkv, T, _ = L.k.shape
    T_cap = _bench_T_cap(T)
    ork, orv = G.oracle_cache(synth.as_float(L.k), synth.as_float(L.v), sets, per_seq, T_cap)
    rk, rv = _encode_gpu(P, L.k, L.v, per_seq, T_cap=T_cap)
    n_diff, n_all = 0.0, 0
    for b in range(B):
        for h in range(Hkv):
            pk, pv = sets[G.set_index(b, h, Hkv, per_seq)]
            for got, ref, p in ((rk[b, h], ork[b, h], pk), (rv[b, h], orv[b, h], pv)):
                nd, na = _compare_records(got, ref, p, T)
                n_diff += nd
                n_all += na
    assert n_diff / n_all <= 1e-4, (n_diff / n_all, round(n_diff), n_all)
    seq = [T] * B
    got = G.run_decode(P, ork, orv, L.q[0], seq, w.Hq, per_seq)
    ref = G.oracle_decode(ork, orv, L.q[0], seq, sets, w.Hq, per_seq)
    err = G.rel_l2_rows(got, ref)
    assert err.max() <= DEC_TOL, err.max()
    return n_diff / n_all, err.max()


@pytest.fixture(scope="module")
def qwen_full():
    w = synth.WORKLOADS["qwen_batched_8k"]
    return w, synth.make_layer(w, steps=1)


@pytest.mark.parametrize("bits", [2.0, 3.0, 4.0])
def test_full_size_qwen_batched_8k(qwen_full, bits):
    """The batched Qwen-shaped workload at full size: 16 sequences x 4 KV heads x 8192 Student-t keys, 7 query
    heads per KV head, one parameter set per (sequence, head) from the sequence's own first 1024 tokens."""
    w, L = qwen_full
    print("entry mismatch %.2e, decode rel-L2 max %.2e" % _full_size_case(w, L, bits))


def test_full_size_llama_long_128k():
    """The long-context workload at full size: 131072 tokens x 8 KV heads at 1.33 bits per element (5-word
    records, most channels at zero width)."""
    w = synth.WORKLOADS["llama_long_128k"]
    L = synth.make_layer(w, steps=1)
    print("entry mismatch %.2e, decode rel-L2 max %.2e" % _full_size_case(w, L, 1.33))


def test_prefill_stack_full_size_sampled():
    """The 32-layer prefill workload at full size. Per layer: tokens drawn on the device (4 sequences x 8 KV
    heads x 65536 bf16 tokens), oracle parameters calibrated on tokens 0..4095 of sequence 0, one kv_encode of
    the whole layer (the tensor-core path), 64 sampled token pairs of every (sequence, head) against the oracle
    encode; then one decode step over the layer's cache. On every fourth layer one (sequence, head)'s records
    are replaced by the oracle's records of all its tokens, and that pair's decode rows are checked against the
    oracle decode."""
    w = synth.WORKLOADS["llama_prefill_32l"]
    B, Hkv, Hq, T, g, d = w.B, w.Hkv, w.Hq, w.T, w.g, w.d
    rng = np.random.default_rng(11)
    scale = 1.0 / math.sqrt(d)
    n_diff, n_all, worst = 0.0, 0, 0.0
    for layer in range(w.layers):
        Ld = synth.make_layer_device(w, layer, "cuda")
        sets = G.calibrate_oracle(Ld, 2.75, 2.75)
        P = G.lib_params(sets)
        Rk, Rv = P.record_words(0), P.record_words(1)
        rk = torch.zeros((B, Hkv, T, Rk), dtype=torch.int32, device="cuda")
        rv = torch.zeros(G.value_cache_shape(B, Hkv, T, Rv), dtype=torch.int32, device="cuda")
        cache = kvtc.make_cache(rk, rv, B, Hkv, T, False)
        kvtc.kv_encode(P, cache, Ld.k, Ld.v, kvtc.KV_DTYPE_BF16, B, T, torch.zeros(B, dtype=torch.int64,
                                                                                      device="cuda"))
        assert kvtc.kv_check_status() == kvtc.KV_OK, kvtc.kv_last_error()
        for b in range(B):
            for h in range(Hkv):
                pk, pv = sets[h]
                pairs = np.sort(rng.choice(T // 2, 64, replace=False))
                toks = np.stack([2 * pairs, 2 * pairs + 1], 1).reshape(-1)
                ti, pi = torch.from_numpy(toks).cuda(), torch.from_numpy(pairs).cuda()
                kx = Ld.k[b, h, ti].double().cpu().numpy()
                vx = Ld.v[b, h, ti].double().cpu().numpy()
                for got, x, p in ((G.u32(rk[b, h, ti]), kx, pk), (G.u32(rv[b, h, pi]), vx, pv)):
                    tf, dz, ds, cf, dc, ef = G.token_diff(O.unpack(got, p), O.unpack(O.encode(x, p), p), p)
                    assert dc <= 1 and dz <= 1 and ds <= 1, (layer, b, h, dz, ds, dc)
                    n = len(toks) * (int(np.count_nonzero(p.widths)) + 2)
                    n_diff += ef * n
                    n_all += n
        check = layer % 4 == 0
        if check:
            bc, hc = int(rng.integers(B)), int(rng.integers(Hkv))
            pk, pv = sets[hc]
            ork = O.encode(Ld.k[bc, hc].double().cpu().numpy(), pk)
            orv = O.encode(Ld.v[bc, hc].double().cpu().numpy(), pv)
            rk[bc, hc] = G.dev_u32(ork)
            rv[bc, hc] = G.dev_u32(orv)
        q = G.to_dev_storage(Ld.q[0])
        sl = torch.full((B,), T, dtype=torch.int32, device="cuda")
        out = torch.full((B, Hq, d), float("nan"), dtype=torch.float32, device="cuda")
        ws = torch.zeros(kvtc.kv_decode_workspace_bytes(P, B, Hkv, Hq, T), dtype=torch.uint8, device="cuda")
        kvtc.kv_attend_decode(P, cache, q, B, Hq, sl, scale, out, ws)
        assert kvtc.kv_check_status() == kvtc.KV_OK, kvtc.kv_last_error()
        o = out.cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(o))
        if check:
            qf = synth.as_float(Ld.q[0])
            ref = O.attend_decode(qf[bc, hc * g:(hc + 1) * g], ork, orv, pk, pv, T, scale)
            err = G.rel_l2_rows(o[bc, hc * g:(hc + 1) * g], ref)
            assert err.max() <= DEC_TOL, (layer, bc, hc, err)
            worst = max(worst, float(err.max()))
        del Ld, rk, rv, cache
    assert n_diff / n_all <= 1e-4, (n_diff / n_all, round(n_diff), n_all)
    print("sampled entry mismatch %.2e, decode rel-L2 max %.2e" % (n_diff / n_all, worst))
