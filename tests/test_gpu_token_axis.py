"""Token-axis allocation on the GPU against the oracle: token weights from the observation queries' attention
(tensor cores), the kept tokens (one-tier reverse water-filling: the heaviest tokens, ties to the earlier one),
record compaction, and the decode over the compacted cache, end to end through the C ABI."""
import math

import numpy as np
import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

from oracle import kvtc_oracle as O  # noqa: E402
from transform_coded_kv_02_b300 import kvtc, synth  # noqa: E402

import gpu_helpers as G  # noqa: E402
from test_gpu_parity import _compare_records  # noqa: E402

DEC_TOL = 2e-3


def _obs_queries(L):
    """The layer's decode queries [W, B, Hq, d] as observation queries [B, Hq, W, d] (bf16 bits)."""
    return np.ascontiguousarray(np.transpose(L.q, (1, 2, 0, 3)))


def _oracle_weights(q_obs_bits, k_bits, Hkv, scale):
    q = synth.as_float(q_obs_bits)
    k = synth.as_float(k_bits)
    B, Hq, W, d = q.shape
    g = Hq // Hkv
    lam = np.zeros(k.shape[:3])
    for b in range(B):
        for h in range(Hkv):
            lam[b, h] = O.token_weights(q[b, h * g:(h + 1) * g].reshape(g * W, d), k[b, h], scale)
    return lam


def _gpu_weights(q_obs_bits, k_bits, Hkv, scale):
    B, Hq, W, d = q_obs_bits.shape
    T = k_bits.shape[2]
    lam = torch.full((B, Hkv, T), float("nan"), dtype=torch.float32, device=G.DEV)
    ws = torch.empty(kvtc.kv_token_weights_workspace_bytes(B, Hkv, T), dtype=torch.uint8, device=G.DEV)
    kvtc.kv_token_weights(G.to_dev_storage(q_obs_bits), W, G.to_dev_storage(k_bits), B, Hkv, Hq, T, scale, lam, ws)
    assert kvtc.kv_check_status() == kvtc.KV_OK, kvtc.kv_last_error()
    return lam


@pytest.mark.parametrize("name,W,T", [("llama_decode_32k", 32, 1000), ("qwen_batched_8k", 16, 777),
                                      ("llama_decode_32k", 5, 130), ("tiny", 32, 1),
                                      ("llama_decode_32k", 32, 20000), ("qwen_batched_8k", 16, 9000)])
def test_token_weights_match_oracle(name, W, T):
    """g x W observation rows (128, 112, 20 and 128 of the MMA's 128), ragged last tiles, one-token sequences.
    The two longer cases hold more tiles than two per SM, so each CTA takes a run of tiles (5 and 2 on 148 SMs) with
    its keys double-buffered, and the last run of a (sequence, KV head) is shorter than the others."""
    w = synth.WORKLOADS[name]
    B = 2 if w.B > 1 else 1
    L = synth.make_layer(w, T=T, steps=W, B=B)
    scale = 1.0 / math.sqrt(128)
    q_obs = _obs_queries(L)
    k = L.k if L.k.dtype == np.uint16 else synth.round_to(L.k, "bf16")  # the weights take bf16 keys
    got = _gpu_weights(q_obs, k, w.Hkv, scale).cpu().numpy().astype(np.float64)
    ref = _oracle_weights(q_obs, k, w.Hkv, scale)
    assert np.all(np.isfinite(got))
    err = np.abs(got - ref)
    assert np.all(err <= 1e-4 * ref + 1e-7 * ref.max()), float((err / np.maximum(ref, 1e-30)).max())
    # each query's probabilities sum to one: sum_t lambda_t lies between n_q / T and n_q
    nq = (w.Hq // w.Hkv) * W
    s = got.sum(axis=2)
    assert np.all(s >= nq / T * (1 - 1e-5)) and np.all(s <= nq * (1 + 1e-5))


def _select_inputs(B, Hkv, T):
    rng = np.random.default_rng(T)
    lam = rng.choice(np.array([0.0, 1e-3, 0.25, 0.5, 0.5, 1.0, 7.0], np.float32), size=(B, Hkv, T))
    lam[0, min(1, Hkv - 1)] = rng.random(T).astype(np.float32)  # one row without ties
    return lam


def _check_select(lam, keeps):
    B, Hkv, T = lam.shape
    lam_dev = torch.from_numpy(lam).to(G.DEV)
    for keep in keeps:
        idx = torch.full((B, Hkv, max(keep, 1)), -7, dtype=torch.int32, device=G.DEV)
        kvtc.kv_token_select(lam_dev, B, Hkv, T, keep, idx)
        assert kvtc.kv_check_status() == kvtc.KV_OK, kvtc.kv_last_error()
        got = idx.cpu().numpy()
        for b in range(B):
            for h in range(Hkv):
                want = O.token_keep(lam[b, h].astype(np.float64), keep)
                assert np.array_equal(got[b, h, :keep], want), (b, h, keep)


@pytest.mark.parametrize("T,keeps", [(1, [0, 1]), (5, [1, 2, 5]), (1000, [1, 333, 999, 1000]),
                                     (5000, [2500, 1]), (60000, [15000, 59999])])
def test_token_select_matches_oracle(T, keeps):
    """Seeded weights with many exact ties and zeros: the kept set equals the oracle's, index for index. Six rows
    take clusters of 8 CTAs on 148 SMs, so the CTAs hold from nothing (1 and 5 tokens) to 7500 tokens each."""
    _check_select(_select_inputs(2, 3, T), keeps)


@pytest.mark.parametrize("B,Hkv,T,keeps", [(5, 8, 3000, [1, 1500, 2999]), (20, 8, 700, [350, 699]),
                                           (1, 1, 400000, [100000, 1])])
def test_token_select_cluster_sizes(B, Hkv, T, keeps):
    """The cluster per (sequence, KV head) is sized to the SMs: on 148 SMs 40 rows take clusters of 2 CTAs and 160
    rows single CTAs; one row of 400000 tokens takes 8 CTAs of 50000 tokens, more than shared memory holds, so
    every pass rereads the weights from global memory."""
    _check_select(_select_inputs(B, Hkv, T), keeps)


def _keep_at_gap(lam_rows, target, rel=1e-3):
    """A keep count near target where every row's keep-th and next weights differ by more than rel: both sides then
    keep the same tokens whatever their rounding."""
    T = lam_rows.shape[-1]
    srt = -np.sort(-lam_rows, axis=-1)
    for off in range(T):
        for keep in (target - off, target + off):
            if 1 <= keep < T:
                a, b = srt[..., keep - 1], srt[..., keep]
                if np.all(a - b > rel * a):
                    return keep
    return T


@pytest.mark.parametrize("keep_frac", [0.25, 0.5])
def test_evict_then_decode_matches_oracle(keep_frac):
    """The whole path on the GPU: encode the prefill, weigh the tokens, keep the heaviest, compact, decode over the
    kept tokens; against the oracle's weights, selection, records and decode. The keep count sits where the
    oracle's weights have a clear gap, so both sides keep the same tokens; an odd count re-pairs value halves.
    The compacted records meet the encode's bar (entries within one step, at most 1e-4 of them off); the decode
    kernel over the oracle's compacted records meets the decode bar; the end-to-end output, whose rare one-step
    record differences sit on the heaviest tokens by construction, is held to ten times the decode bar."""
    w = synth.WORKLOADS["llama_decode_32k"]
    B, T, W, T_cap = 2, 900, 32, 912
    L = synth.make_layer(w, T=T, steps=W + 1, B=B)  # W observation queries, then the decode query
    sets = G.calibrate_oracle(L, 2.75, 2.75)
    P = G.lib_params(sets)
    scale = 1.0 / math.sqrt(128)
    q_obs = np.ascontiguousarray(np.transpose(L.q[:W], (1, 2, 0, 3)))
    lam_o = _oracle_weights(q_obs, L.k, w.Hkv, scale)
    keep = _keep_at_gap(lam_o, int(keep_frac * T) | 1)
    # device path
    Rk, Rv = sets[0][0].r_words, sets[0][1].r_words
    rk = torch.zeros((B, w.Hkv, T_cap, Rk), dtype=torch.int32, device=G.DEV)
    rv = torch.zeros((B, w.Hkv, T_cap // 2, 2 * Rv), dtype=torch.int32, device=G.DEV)
    src = kvtc.make_cache(rk, rv, B, w.Hkv, T_cap)
    kvtc.kv_encode(P, src, G.to_dev_storage(L.k), G.to_dev_storage(L.v), kvtc.KV_DTYPE_BF16, B, T,
                   torch.zeros(B, dtype=torch.int64, device=G.DEV))
    lam = _gpu_weights(q_obs, L.k, w.Hkv, scale)
    idx = torch.empty((B, w.Hkv, keep), dtype=torch.int32, device=G.DEV)
    kvtc.kv_token_select(lam, B, w.Hkv, T, keep, idx)
    ck = torch.zeros((B, w.Hkv, T_cap, Rk), dtype=torch.int32, device=G.DEV)
    cv = torch.zeros((B, w.Hkv, T_cap // 2, 2 * Rv), dtype=torch.int32, device=G.DEV)
    dst = kvtc.make_cache(ck, cv, B, w.Hkv, T_cap)
    kvtc.kv_cache_compact(P, src, dst, B, idx, keep)
    q = G.to_dev_storage(L.q[W])
    out = torch.full((B, w.Hq, 128), float("nan"), dtype=torch.float32, device=G.DEV)
    ws = torch.zeros(kvtc.kv_decode_workspace_bytes(P, B, w.Hkv, w.Hq, T_cap), dtype=torch.uint8, device=G.DEV)
    kvtc.kv_attend_decode(P, dst, q, B, w.Hq, torch.full((B,), keep, dtype=torch.int32, device=G.DEV), scale, out, ws)
    assert kvtc.kv_check_status() == kvtc.KV_OK, kvtc.kv_last_error()
    # oracle path
    k, v = synth.as_float(L.k), synth.as_float(L.v)
    got_idx = idx.cpu().numpy()
    ork = np.zeros((B, w.Hkv, T_cap, Rk), np.uint32)
    orv = np.zeros((B, w.Hkv, T_cap // 2, 2 * Rv), np.uint32)
    for b in range(B):
        for h in range(w.Hkv):
            kept = O.token_keep(lam_o[b, h], keep)
            assert np.array_equal(got_idx[b, h], kept), (b, h)
            pk, pv = sets[h]
            ork[b, h, :keep] = O.compact(O.encode(k[b, h], pk), pk, kept)
            orv[b, h, :(keep + 1) // 2] = O.compact(O.encode(v[b, h], pv), pv, kept)
    gk, gv = G.u32(ck), G.u32(cv)
    n_diff, n_all = 0.0, 0
    for b in range(B):
        for h in range(w.Hkv):
            pk, pv = sets[h]
            for got_r, ref_r, p in ((gk[b, h], ork[b, h], pk), (gv[b, h], orv[b, h], pv)):
                nd, na = _compare_records(got_r, ref_r, p, keep)
                n_diff += nd
                n_all += na
    assert n_diff / n_all <= 1e-4, (n_diff, n_all)
    ref = G.oracle_decode(ork, orv, L.q[W], [keep] * B, sets, w.Hq, False)
    kern = G.run_decode(P, ork, orv, L.q[W], [keep] * B, w.Hq, False)
    assert G.rel_l2_rows(kern, ref).max() <= DEC_TOL
    err = G.rel_l2_rows(out.cpu().numpy().astype(np.float64), ref)
    assert err.max() <= 10 * DEC_TOL, err.max()


@pytest.mark.parametrize("keep", [1, 2, 37, 300])
def test_compact_matches_oracle(keep):
    """Compaction of the oracle's records by a seeded selection equals the oracle's compaction, bit for bit; the
    destination's other records stay untouched."""
    w = synth.WORKLOADS["qwen_batched_8k"]
    B, T, T_cap = 2, 300, 320
    L = synth.make_layer(w, T=T, steps=1, B=B)
    sets = G.calibrate_oracle(L, 3.0, 3.0)
    P = G.lib_params(sets)
    rk, rv = G.oracle_cache(synth.as_float(L.k), synth.as_float(L.v), sets, True, T_cap)
    rng = np.random.default_rng(keep)
    sel = np.stack([np.stack([np.sort(rng.choice(T, keep, replace=False)) for _ in range(w.Hkv)])
                    for _ in range(B)]).astype(np.int32)
    sk, sv = G.dev_u32(rk), G.dev_u32(rv)  # (kept alive: the cache struct holds raw pointers)
    src = kvtc.make_cache(sk, sv, B, w.Hkv, T_cap, True)
    dk = torch.full((B, w.Hkv, T_cap, rk.shape[-1]), 0x5A5A5A5A, dtype=torch.int32, device=G.DEV)
    dv = torch.full((B, w.Hkv, T_cap // 2, rv.shape[-1]), 0x5A5A5A5A, dtype=torch.int32, device=G.DEV)
    dst = kvtc.make_cache(dk, dv, B, w.Hkv, T_cap, True)
    kvtc.kv_cache_compact(P, src, dst, B, torch.from_numpy(sel).to(G.DEV), keep)
    assert kvtc.kv_check_status() == kvtc.KV_OK, kvtc.kv_last_error()
    gk, gv = G.u32(dk), G.u32(dv)
    for b in range(B):
        for h in range(w.Hkv):
            pk, pv = sets[G.set_index(b, h, w.Hkv, True)]
            assert np.array_equal(gk[b, h, :keep], O.compact(rk[b, h], pk, sel[b, h]))
            assert np.array_equal(gv[b, h, :(keep + 1) // 2], O.compact(rv[b, h], pv, sel[b, h]))
            assert np.all(gk[b, h, keep:] == 0x5A5A5A5A) and np.all(gv[b, h, (keep + 1) // 2:] == 0x5A5A5A5A)
