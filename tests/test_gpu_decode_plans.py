"""Decode over every launch plan the device offers. The splits of one (sequence, KV head) merge either inside a
thread-block cluster of 16, 8, 4, 2 or 1 CTAs, through distributed shared memory, or through the workspace, the
last split to arrive doing the merge. B * Hkv, the SM count and how many clusters of each size the device holds at
once decide the plan: kv_debug_decode_plan reports it without launching, and the shapes below are searched for
each plan. Every case is checked against the oracle decode over the same records (the oracle's), with ragged
sequence lengths."""
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

DEC_TOL = 2e-3  # relative L2 per output row against the exact decode of the same records


def _one_set_params(w, bits):
    L = synth.make_layer(w, T=256, steps=1, B=1)
    sets = G.calibrate_oracle(L, bits, bits)
    return sets, G.lib_params(sets)


def _batch_for_plan(P, Hkv, Hq, T_cap, want, b_max=160):
    for B in range(1, b_max + 1):
        plan = kvtc.kv_debug_decode_plan(P, B, Hkv, Hq, T_cap)
        if plan["cluster"] == want:
            return B, plan
    return None, None


@pytest.mark.parametrize("want", [16, 8, 4, 2, 1, 0])
def test_decode_every_cluster_size_one_head_per_sequence(want):
    """One KV head of four query heads per sequence (the tiny workload's shape) and B sequences, B picked so that
    the decode takes the wanted plan: cluster size 16, 8, 4, 2, 1, or 0 (the workspace merge)."""
    w = synth.WORKLOADS["tiny"]
    sets, P = _one_set_params(w, 2.75)
    T, T_cap = 300, 320
    B, plan = _batch_for_plan(P, 1, w.Hq, T_cap, want)
    if B is None:
        pytest.skip(f"this device offers no plan with cluster size {want} for one KV head per sequence")
    Lb = synth.make_layer(w, T=T, steps=1, B=B)
    k, v = synth.as_float(Lb.k), synth.as_float(Lb.v)
    rk, rv = G.oracle_cache(k, v, sets, False, T_cap)
    seq = [max(1, T - (37 * b) % 290) for b in range(B)]
    got = G.run_decode(P, rk, rv, Lb.q[0], seq, w.Hq, False)
    ref = G.oracle_decode(rk, rv, Lb.q[0], seq, sets, w.Hq, False)
    err = G.rel_l2_rows(got, ref)
    assert np.all(np.isfinite(got))
    assert err.max() <= DEC_TOL, (B, plan, err.max())


@pytest.mark.parametrize("want", [4, 2])
def test_decode_cluster_two_column_blocks_per_sequence_sets(want):
    """Seven query heads per KV head (two column blocks, eight warps) with a parameter set per (sequence, head),
    in a cluster of 4 or 2."""
    w = synth.WORKLOADS["qwen_batched_8k"]
    T, T_cap = 256, 256
    probe = synth.make_layer(w, T=T, steps=1, B=1)
    P0 = G.lib_params(G.calibrate_oracle(probe, 3.0, 3.0))
    B, plan = _batch_for_plan(P0, w.Hkv, w.Hq, T_cap, want, b_max=40)
    if B is None:
        pytest.skip(f"this device offers no plan with cluster size {want} for this shape")
    Lb = synth.make_layer(w, T=T, steps=1, B=B)
    sets = G.calibrate_oracle(Lb, 3.0, 3.0)
    P = G.lib_params(sets)
    k, v = synth.as_float(Lb.k), synth.as_float(Lb.v)
    rk, rv = G.oracle_cache(k, v, sets, True, T_cap)
    seq = [max(1, T - (53 * b) % 250) for b in range(B)]
    got = G.run_decode(P, rk, rv, Lb.q[0], seq, w.Hq, True)
    ref = G.oracle_decode(rk, rv, Lb.q[0], seq, sets, w.Hq, True)
    err = G.rel_l2_rows(got, ref)
    assert err.max() <= DEC_TOL, (B, plan, err.max())


def test_decode_plan_reports_a_consistent_launch():
    """The plan's fields agree with each other: a cluster plan has as many splits as CTAs in its cluster and the
    device holds all B * Hkv clusters at once; the shared memory fits a CTA."""
    w = synth.WORKLOADS["tiny"]
    _, P = _one_set_params(w, 2.75)
    for B in (1, 4, 6, 12, 24, 48, 100, 200):
        plan = kvtc.kv_debug_decode_plan(P, B, 1, w.Hq, 1024)
        assert plan["warps"] in (8, 16) and plan["channel_blocks"] in (4, 8)
        assert 0 < plan["smem_bytes"] <= 227 * 1024
        assert plan["stages"] >= 2
        if plan["cluster"] > 0:
            assert plan["splits"] == plan["cluster"]
            held = plan["clusters_held"][plan["cluster"]]
            assert held >= B or plan["cluster"] == 1
        else:
            assert plan["splits"] >= 1


def _with_widths(p, width, n_channels):
    """The oracle table p with its first n_channels channels at one width and the rest at zero."""
    w = np.zeros(p.d, np.int64)
    w[:n_channels] = width
    return O.TensorParams(T=p.T, mu=p.mu, sigma=p.sigma, widths=w, r_words=p.r_words, pairing=p.pairing)


# (key pair-slot width, value slot width) -> channels of that width that fill the 7 key code words / 14 value half
# words of 8-word records, and whether every lane's two slots of a block the decode reads can share one word: an
# even number of slots per word (width 2 or 4) couples within words; an odd number (3 or 5) leaves one slot per word
# that, without enough zero-width partners in the blocks read, pairs with a slot of another word
_FILL = {2: (112, 112, True), 3: (70, 70, False), 4: (56, 56, True), 5: (42, 42, False)}


@pytest.mark.parametrize("name", ["llama_decode_32k", "qwen_batched_8k"])
@pytest.mark.parametrize("wk,wv", [(4, 4), (5, 4), (4, 5), (5, 5), (2, 2), (3, 3), (2, 3), (3, 2)])
def test_decode_single_word_variants(name, wk, wv):
    """Tables whose key and value blocks do, or do not, hold each lane's two slots in one code word: the decode
    takes the kernel without the per-block test for the tensors where every set allows it (single_word bit 0:
    keys, bit 1: values), and matches the oracle decode either way. Widths are set by hand on 8-word records (a
    compiled record length); four or eight channel blocks as the channels need."""
    w = synth.WORKLOADS[name]
    B = 2 if w.calib == "own_prefix" else 1
    T, T_cap = 700, 704
    L = synth.make_layer(w, T=T, steps=1, B=B)
    base = [O.calibrate(ck, cv, cq, 2.0, 2.0) for ck, cv, cq in zip(L.calib_k, L.calib_v, L.calib_q)]
    assert base[0][0].r_words == 8 and base[0][1].r_words == 8
    (nk, _, sk), (_, nv, sv) = _FILL[wk], _FILL[wv]
    sets = [(_with_widths(pk, wk, nk), _with_widths(pv, wv, nv)) for pk, pv in base]
    P = G.lib_params(sets)
    per_seq = L.per_seq_params
    plan = kvtc.kv_debug_decode_plan(P, B, w.Hkv, w.Hq, T_cap)
    assert plan["single_word"] == (1 if sk else 0) | (2 if sv else 0), plan
    assert plan["channel_blocks"] == (4 if max(nk, nv) <= 64 else 8)
    k, v = synth.as_float(L.k), synth.as_float(L.v)
    rk, rv = G.oracle_cache(k, v, sets, per_seq, T_cap)
    seq = [T, 433][:B]
    got = G.run_decode(P, rk, rv, L.q[0], seq, w.Hq, per_seq)
    ref = G.oracle_decode(rk, rv, L.q[0], seq, sets, w.Hq, per_seq)
    err = G.rel_l2_rows(got, ref)
    assert np.all(np.isfinite(got))
    assert err.max() <= DEC_TOL, (plan, err.max())
