"""Paged, multi-layer decode and encode in one launch, and the query's rotary embedding in the decode kernel, all
through the C ABI and against the oracle. Records live in page pools [n_pages][Hkv][P][R] reached through a block
table per (layer, sequence); the pages of a sequence are scattered at random over the pool, and table entries past a
sequence's length are out of range (-1), which a read of them would report. Each layer has its own parameter sets
(one table over every layer's heads, layer-major)."""
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

DEC_TOL = 2e-3   # relative L2 per output row against the exact decode of the same records
ROPE_BASE = 500000.0


def _layers(w, n_layers, T, B, bits):
    """Per layer: synthetic data and the oracle's sets (per head, or per (sequence, head))."""
    out = []
    for layer in range(n_layers):
        L = synth.make_layer(w, layer=layer, T=T, steps=1, B=B)
        out.append((L, G.calibrate_oracle(L, bits, bits)))
    return out


def _page_tables(rng, n_z, seq_lens_z, P, max_pages, spare=5):
    """A block table [n_z][max_pages] giving every page a sequence reads a distinct pool page, in random order;
    entries past the sequence's pages are -1."""
    need = [(-(-int(n) // P)) for n in seq_lens_z]
    n_pages = sum(need) + spare
    perm = rng.permutation(n_pages)
    bt = np.full((n_z, max_pages), -1, np.int32)
    k = 0
    for z in range(n_z):
        for i in range(need[z]):
            bt[z, i] = perm[k]
            k += 1
    return bt, n_pages


def _scatter(rk, rv, bt, n_pages, P):
    """Dense records rk [Z, Hkv, T_cap, Rk], rv [Z, Hkv, T_cap / 2, 2 Rv] -> page pools by the block table."""
    Z, Hkv, _, Rk = rk.shape
    Rv2 = rv.shape[-1]
    kp = np.zeros((n_pages, Hkv, P, Rk), np.uint32)
    vp = np.zeros((n_pages, Hkv, P // 2, Rv2), np.uint32)
    for z in range(Z):
        for i, pg in enumerate(bt[z]):
            if pg < 0:
                continue
            kp[pg] = rk[z, :, i * P:(i + 1) * P]
            vp[pg] = rv[z, :, i * P // 2:(i + 1) * P // 2]
    return kp, vp


def _gather(kp, vp, bt, z, P, n_tokens):
    """The records of virtual sequence z from the pools: keys [n, Rk], values [ceil(n / 2), 2 Rv]."""
    pages = [bt[z, i] for i in range(-(-n_tokens // P))]
    k = np.concatenate([kp[pg] for pg in pages], axis=1)  # [Hkv, pages * P, Rk]
    v = np.concatenate([vp[pg] for pg in pages], axis=1)
    return k, v


def _run_paged_decode(P_lib, kp, vp, bt, n_pages, P, B, n_layers, Hkv, Hq, q_bits, seq, q_pos, per_seq,
                      first_layer=0):
    d = 128
    tkp, tvp = G.dev_u32(kp), G.dev_u32(vp)
    tbt = torch.from_numpy(np.ascontiguousarray(bt)).to(G.DEV)
    cache = kvtc.make_paged_cache(tkp, tvp, n_pages, P, Hkv, B, n_layers, bt.shape[1], tbt, per_seq, first_layer)
    q = G.to_dev_storage(q_bits)
    sl = torch.tensor(seq, dtype=torch.int32, device=G.DEV)
    qp = None if q_pos is None else torch.tensor(q_pos, dtype=torch.int32, device=G.DEV)
    out = torch.full((n_layers, B, Hq, d), float("nan"), dtype=torch.float32, device=G.DEV)
    ws = torch.zeros(kvtc.kv_decode_paged_workspace_bytes(P_lib, cache, Hq), dtype=torch.uint8, device=G.DEV)
    kvtc.kv_attend_decode_paged(P_lib, cache, q, Hq, sl, qp, 1.0 / math.sqrt(d), out, ws)
    st = kvtc.kv_check_status()
    return out.cpu().numpy().astype(np.float64), st


def _oracle(layers, dense, q_bits, seq, q_pos, Hkv, Hq, per_seq, n_layers, B):
    g = Hq // Hkv
    scale = 1.0 / math.sqrt(128)
    ref = np.zeros((n_layers, B, Hq, 128))
    for layer in range(n_layers):
        rk, rv = dense[layer]
        sets = layers[layer][1]
        q = synth.as_float(q_bits[layer])
        for b in range(B):
            for h in range(Hkv):
                pk, pv = sets[G.set_index(b, h, Hkv, per_seq)]
                qh = q[b, h * g:(h + 1) * g]
                if q_pos is not None:
                    qh = O.rotary_embed(qh, int(q_pos[b]), ROPE_BASE)
                ref[layer, b, h * g:(h + 1) * g] = O.attend_decode(qh, rk[b, h], rv[b, h], pk, pv, int(seq[b]), scale)
    return ref


@pytest.mark.parametrize("rope", [False, True])
@pytest.mark.parametrize("name,bits,P", [("llama_decode_32k", 2.75, 32), ("llama_decode_32k", 2.75, 256),
                                         ("qwen_batched_8k", 3.0, 64)])
def test_paged_multi_layer_decode_matches_oracle(name, bits, P, rope):
    """Two layers of B ragged sequences in one launch over scattered pages, with or without the query's rotary
    embedding (positions up to 100000, where an fp32 angle would be off by whole hundredths of a radian)."""
    w = synth.WORKLOADS[name]
    n_layers, T = 2, 700
    B = 3 if not w.calib == "own_prefix" else 2
    T_cap = 768
    layers = _layers(w, n_layers, T, B, bits)
    per_seq = layers[0][0].per_seq_params
    all_sets = [s for _, sets in layers for s in sets]
    P_lib = G.lib_params(all_sets)
    if rope:
        P_lib.set_rope(ROPE_BASE).upload()
    seq = [700, 433, 61][:B]
    q_pos = [699, 100000, 5][:B] if rope else None
    dense = []
    for L, sets in layers:
        dense.append(G.oracle_cache(synth.as_float(L.k), synth.as_float(L.v), sets, per_seq, T_cap))
    rk = np.concatenate([d[0] for d in dense])  # [n_layers * B, Hkv, T_cap, Rk]
    rv = np.concatenate([d[1] for d in dense])
    rng = np.random.default_rng(17 + P)
    max_pages = T_cap // P
    bt, n_pages = _page_tables(rng, n_layers * B, seq * n_layers, P, max_pages)
    kp, vp = _scatter(rk, rv, bt, n_pages, P)
    q_bits = np.stack([L.q[0] for L, _ in layers])  # [n_layers, B, Hq, d]
    got, st = _run_paged_decode(P_lib, kp, vp, bt, n_pages, P, B, n_layers, w.Hkv, w.Hq, q_bits, seq, q_pos,
                                per_seq)
    assert st == kvtc.KV_OK, kvtc.kv_last_error()
    ref = _oracle(layers, dense, q_bits, seq, q_pos, w.Hkv, w.Hq, per_seq, n_layers, B)
    err = G.rel_l2_rows(got, ref)
    assert np.all(np.isfinite(got))
    assert err.max() <= DEC_TOL, err.max()
    if rope:  # the embedding matters at these positions: without it the result is far off
        plain = _oracle(layers, dense, q_bits, seq, None, w.Hkv, w.Hq, per_seq, n_layers, B)
        assert G.rel_l2_rows(got, plain).max() > 10 * DEC_TOL


def test_paged_view_of_one_layer():
    """A view of layer 1 alone (its block-table rows, first_layer = 1) decodes that layer with its own sets."""
    w = synth.WORKLOADS["llama_decode_32k"]
    T, T_cap, B, P = 500, 512, 2, 64
    layers = _layers(w, 2, T, B, 2.75)
    P_lib = G.lib_params([s for _, sets in layers for s in sets])
    seq = [500, 130]
    dense = [G.oracle_cache(synth.as_float(L.k), synth.as_float(L.v), sets, False, T_cap) for L, sets in layers]
    rng = np.random.default_rng(3)
    bt, n_pages = _page_tables(rng, B, seq, P, T_cap // P)
    kp, vp = _scatter(dense[1][0], dense[1][1], bt, n_pages, P)
    q_bits = layers[1][0].q[0][None]
    got, st = _run_paged_decode(P_lib, kp, vp, bt, n_pages, P, B, 1, w.Hkv, w.Hq, q_bits, seq, None, False,
                                first_layer=1)
    assert st == kvtc.KV_OK, kvtc.kv_last_error()
    ref = _oracle([layers[1]], [dense[1]], q_bits, seq, None, w.Hkv, w.Hq, False, 1, B)
    assert G.rel_l2_rows(got, ref).max() <= DEC_TOL


def _dense_encode(P_lib, k_dev, v_dev, dtype, B, Hkv, T_cap, t_new, pos, per_seq, Rk, Rv):
    rk = torch.zeros((B, Hkv, T_cap, Rk), dtype=torch.int32, device=G.DEV)
    rv = torch.zeros((B, Hkv, T_cap // 2, 2 * Rv), dtype=torch.int32, device=G.DEV)
    cache = kvtc.make_cache(rk, rv, B, Hkv, T_cap, per_seq)
    kvtc.kv_encode(P_lib, cache, k_dev, v_dev, dtype, B, t_new, pos)
    return rk, rv


@pytest.mark.parametrize("path", [0, 1])
def test_paged_encode_matches_dense_and_oracle(path):
    """Prefill (300 bf16 tokens: the tensor cores on path 0, CUDA cores on path 1), then appends of one and of
    three tokens at odd and even positions, into scattered pages of two layers in one launch each. Every record
    equals the one the dense cache gets from the same kernel (layer by layer), and matches the oracle."""
    w = synth.WORKLOADS["llama_decode_32k"]
    n_layers, B, Hkv, P, T_cap = 2, 2, w.Hkv, 64, 512
    T0, steps = 300, [1, 3, 1]
    T = T0 + sum(steps)
    layers = _layers(w, n_layers, T, B, 2.75)
    sets_all = [s for _, sets in layers for s in sets]
    P_lib = G.lib_params(sets_all)
    Rk, Rv = sets_all[0][0].r_words, sets_all[0][1].r_words
    rng = np.random.default_rng(11)
    bt, n_pages = _page_tables(rng, n_layers * B, [T_cap] * (n_layers * B), P, T_cap // P)
    kp = torch.zeros((n_pages, Hkv, P, Rk), dtype=torch.int32, device=G.DEV)
    vp = torch.zeros((n_pages, Hkv, P // 2, 2 * Rv), dtype=torch.int32, device=G.DEV)
    tbt = torch.from_numpy(bt).to(G.DEV)
    cache = kvtc.make_paged_cache(kp, vp, n_pages, P, Hkv, B, n_layers, bt.shape[1], tbt, False, 0)
    kvtc.kv_debug_set_encode_path(path)
    try:
        dense = [[None, None] for _ in range(n_layers)]
        t = 0
        for n in [T0] + steps:
            pos = torch.tensor([t, t + 5][:B], dtype=torch.int64, device=G.DEV)  # sequences at different offsets
            kl = np.stack([L.k[:, :, t:t + n] for L, _ in layers])  # [n_layers, B, Hkv, n, d] bf16 bits
            vl = np.stack([L.v[:, :, t:t + n] for L, _ in layers])
            kvtc.kv_encode_paged(P_lib, cache, G.to_dev_storage(np.ascontiguousarray(kl)),
                                 G.to_dev_storage(np.ascontiguousarray(vl)), kvtc.KV_DTYPE_BF16, n, pos)
            for layer in range(n_layers):  # the same tokens, one layer at a time, into dense caches
                view = [s for s in layers[layer][1]]
                P_one = G.lib_params(view)
                if dense[layer][0] is None:
                    dense[layer] = list(_dense_encode(P_one, G.to_dev_storage(np.ascontiguousarray(kl[layer])),
                                                      G.to_dev_storage(np.ascontiguousarray(vl[layer])),
                                                      kvtc.KV_DTYPE_BF16, B, Hkv, T_cap, n, pos, False, Rk, Rv))
                else:
                    c1 = kvtc.make_cache(dense[layer][0], dense[layer][1], B, Hkv, T_cap, False)
                    kvtc.kv_encode(P_one, c1, G.to_dev_storage(np.ascontiguousarray(kl[layer])),
                                   G.to_dev_storage(np.ascontiguousarray(vl[layer])), kvtc.KV_DTYPE_BF16, B, n, pos)
            t += n
        assert kvtc.kv_check_status() == kvtc.KV_OK, kvtc.kv_last_error()
    finally:
        kvtc.kv_debug_set_encode_path(0)
    kp_h = G.u32(kp)
    vp_h = G.u32(vp)
    for layer in range(n_layers):
        rk_d, rv_d = G.u32(dense[layer][0]), G.u32(dense[layer][1])
        L, sets = layers[layer]
        for b in range(B):
            z = layer * B + b
            n_tok = T + 5 * b
            gk, gv = _gather(kp_h, vp_h, bt, z, P, n_tok)
            assert np.array_equal(gk[:, :n_tok], rk_d[b, :, :n_tok]), (layer, b)
            assert np.array_equal(gv[:, :(n_tok + 1) // 2], rv_d[b, :, :(n_tok + 1) // 2]), (layer, b)
            for h in range(Hkv):  # and against the oracle's records of the same tokens
                pk, pv = sets[h]
                lo = 5 * b
                ork = O.encode(synth.as_float(L.k[b, h, :T]), pk)
                _, _, _, fk, _, _ = G.code_diff(gk[h, lo:lo + T], ork, pk)
                assert fk <= 2e-3, (layer, b, h, fk)


def test_paged_bad_page_is_reported():
    """A block-table entry out of range inside a sequence's pages: the decode leaves those tokens out, returns,
    and kv_check_status reports KV_ERR_DEVICE; the next call with a good table is clean."""
    w = synth.WORKLOADS["tiny"]
    T, T_cap, P = 200, 256, 32
    layers = _layers(w, 1, T, 1, 2.75)
    L, sets = layers[0]
    P_lib = G.lib_params(sets)
    rk, rv = G.oracle_cache(synth.as_float(L.k), synth.as_float(L.v), sets, False, T_cap)
    bt, n_pages = _page_tables(np.random.default_rng(1), 1, [T], P, T_cap // P)
    kp, vp = _scatter(rk, rv, bt, n_pages, P)
    bad = bt.copy()
    bad[0, 2] = n_pages + 7
    _, st = _run_paged_decode(P_lib, kp, vp, bad, n_pages, P, 1, 1, w.Hkv, w.Hq, L.q[0][None], [T], None, False)
    assert st == kvtc.KV_ERR_DEVICE
    got, st = _run_paged_decode(P_lib, kp, vp, bt, n_pages, P, 1, 1, w.Hkv, w.Hq, L.q[0][None], [T], None, False)
    assert st == kvtc.KV_OK
    ref = _oracle(layers, [(rk, rv)], L.q[0][None], [T], None, w.Hkv, w.Hq, False, 1, 1)
    assert G.rel_l2_rows(got, ref).max() <= DEC_TOL


def test_query_positions_need_a_rope_table():
    w = synth.WORKLOADS["tiny"]
    layers = _layers(w, 1, 64, 1, 2.75)
    P_lib = G.lib_params(layers[0][1])
    rk, rv = G.oracle_cache(synth.as_float(layers[0][0].k), synth.as_float(layers[0][0].v), layers[0][1], False, 64)
    bt, n_pages = _page_tables(np.random.default_rng(2), 1, [64], 32, 2)
    kp, vp = _scatter(rk, rv, bt, n_pages, 32)
    with pytest.raises(kvtc.KvError) as e:
        _run_paged_decode(P_lib, kp, vp, bt, n_pages, 32, 1, 1, w.Hkv, w.Hq, layers[0][0].q[0][None], [64], [63],
                          False)
    assert e.value.status == kvtc.KV_ERR_INVALID_ARG


@pytest.mark.parametrize("kind", ["joint_14_8", "runtime_32_words"])
def test_paged_decode_other_record_lengths(kind):
    """Record lengths beyond the equal-budget kernels through the paged path: the joint split's 14 key and 8 value
    words (a compile-time kernel of unequal lengths) and 8 bits per element, 32 words per token (the kernel that reads
    the lengths at run time); 64-token pages, two layers, rotary embedding on."""
    w = synth.WORKLOADS["llama_decode_32k"]
    n_layers, B, T, T_cap, P = 2, 1, 600, 640, 64
    layers = []
    for layer in range(n_layers):
        L = synth.make_layer(w, layer=layer, T=T, steps=1, B=B)
        if kind == "joint_14_8":
            sets = O.calibrate_joint(list(zip(L.calib_k, L.calib_v, L.calib_q)), 2.75, 2.75)
            assert (sets[0][0].r_words, sets[0][1].r_words) == (14, 8)
        else:
            sets = G.calibrate_oracle(L, 8.0, 8.0)
            assert sets[0][0].r_words == 32
        layers.append((L, sets))
    P_lib = G.lib_params([s for _, sets in layers for s in sets])
    P_lib.set_rope(ROPE_BASE).upload()
    dense = [G.oracle_cache(synth.as_float(L.k), synth.as_float(L.v), sets, False, T_cap) for L, sets in layers]
    rk = np.concatenate([d[0] for d in dense])
    rv = np.concatenate([d[1] for d in dense])
    seq, q_pos = [T], [4321]
    bt, n_pages = _page_tables(np.random.default_rng(9), n_layers * B, seq * n_layers, P, T_cap // P)
    kp, vp = _scatter(rk, rv, bt, n_pages, P)
    q_bits = np.stack([L.q[0] for L, _ in layers])
    got, st = _run_paged_decode(P_lib, kp, vp, bt, n_pages, P, B, n_layers, w.Hkv, w.Hq, q_bits, seq, q_pos, False)
    assert st == kvtc.KV_OK, kvtc.kv_last_error()
    ref = _oracle(layers, dense, q_bits, seq, q_pos, w.Hkv, w.Hq, False, n_layers, B)
    assert G.rel_l2_rows(got, ref).max() <= DEC_TOL


def test_paged_serving_loop_appends_then_decodes():
    """A serving loop over a paged cache: prefill 300 tokens into pages, then eight steps that each append one token
    per sequence (kv_encode_paged, t_new = 1, odd and even positions) and decode over the grown context with the
    query's rotary embedding at its position; every step's output against the oracle over the oracle's records of the
    same tokens, and the appended records against the oracle's."""
    w = synth.WORKLOADS["qwen_batched_8k"]
    B, T0, steps, P, T_cap = 2, 300, 8, 32, 320
    L = synth.make_layer(w, T=T0 + steps, steps=steps, B=B)
    sets = G.calibrate_oracle(L, 3.0, 3.0)
    per_seq = L.per_seq_params
    P_lib = G.lib_params(sets)
    P_lib.set_rope(ROPE_BASE).upload()
    Rk, Rv = sets[0][0].r_words, sets[0][1].r_words
    bt, n_pages = _page_tables(np.random.default_rng(4), B, [T_cap] * B, P, T_cap // P)
    kp = torch.zeros((n_pages, w.Hkv, P, Rk), dtype=torch.int32, device=G.DEV)
    vp = torch.zeros((n_pages, w.Hkv, P // 2, 2 * Rv), dtype=torch.int32, device=G.DEV)
    tbt = torch.from_numpy(bt).to(G.DEV)
    cache = kvtc.make_paged_cache(kp, vp, n_pages, P, w.Hkv, B, 1, bt.shape[1], tbt, per_seq, 0)
    kvtc.kv_encode_paged(P_lib, cache, G.to_dev_storage(np.ascontiguousarray(L.k[:, :, :T0])),
                         G.to_dev_storage(np.ascontiguousarray(L.v[:, :, :T0])), kvtc.KV_DTYPE_BF16, T0,
                         torch.zeros(B, dtype=torch.int64, device=G.DEV))
    k, v = synth.as_float(L.k), synth.as_float(L.v)
    out = torch.zeros((1, B, w.Hq, 128), dtype=torch.float32, device=G.DEV)
    ws = torch.zeros(kvtc.kv_decode_paged_workspace_bytes(P_lib, cache, w.Hq), dtype=torch.uint8, device=G.DEV)
    scale = 1.0 / math.sqrt(128)
    g = w.Hq // w.Hkv
    for i in range(steps):
        t = T0 + i
        kvtc.kv_encode_paged(P_lib, cache, G.to_dev_storage(np.ascontiguousarray(L.k[:, :, t:t + 1])),
                             G.to_dev_storage(np.ascontiguousarray(L.v[:, :, t:t + 1])), kvtc.KV_DTYPE_BF16, 1,
                             torch.full((B,), t, dtype=torch.int64, device=G.DEV))
        q = G.to_dev_storage(L.q[i][None])
        kvtc.kv_attend_decode_paged(P_lib, cache, q, w.Hq, torch.full((B,), t + 1, dtype=torch.int32, device=G.DEV),
                                    torch.full((B,), t, dtype=torch.int32, device=G.DEV), scale, out, ws)
        assert kvtc.kv_check_status() == kvtc.KV_OK, kvtc.kv_last_error()
        got = out.cpu().numpy()[0].astype(np.float64)
        for b in range(B):
            for h in range(w.Hkv):
                pk, pv = sets[G.set_index(b, h, w.Hkv, per_seq)]
                ork, orv = O.encode(k[b, h, :t + 1], pk), O.encode(v[b, h, :t + 1], pv)
                qh = O.rotary_embed(synth.as_float(L.q[i, b, h * g:(h + 1) * g]), t, ROPE_BASE)
                ref = O.attend_decode(qh, ork, orv, pk, pv, t + 1, scale)
                assert G.rel_l2_rows(got[b, h * g:(h + 1) * g], ref).max() <= 5 * DEC_TOL, (i, b, h)
    # the appended tokens' records against the oracle's (keys one per token; values in their two-token records)
    kp_h, vp_h = G.u32(kp), G.u32(vp)
    for b in range(B):
        gk, gv = _gather(kp_h, vp_h, bt, b, P, T0 + steps)
        for h in range(w.Hkv):
            pk, pv = sets[G.set_index(b, h, w.Hkv, per_seq)]
            ork = O.encode(k[b, h, :T0 + steps], pk)
            _, _, _, fk, dk, _ = G.code_diff(gk[h, T0:T0 + steps], ork[T0:T0 + steps], pk)
            assert dk <= 1 and fk <= 2e-2, (b, h, fk)
