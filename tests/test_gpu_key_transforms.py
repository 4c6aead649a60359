"""The two key transforms beyond the KLT through the CUDA path: the attention-aware orthogonal key basis
(oracle `calibrate(..., attention_aware_keys=True)`, the library's key_basis 1) and [NOVA-KV]'s non-orthogonal
key transform (oracle `calibrate(..., whitened_keys=True)`, the library's key_basis 2), whose decode rotates q by
T^-T and forms its folded vectors with T^-1. Parameters come from the oracle and reach the library by
kv_params_from_arrays (with the inverse for the non-orthogonal transform); the encode is checked against the
oracle's records and the decode, over the oracle's records, against the oracle decode."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

from oracle import kvtc_oracle as O  # noqa: E402
from transform_coded_kv_02_b300 import kvtc, synth  # noqa: E402

import gpu_helpers as G  # noqa: E402
from test_gpu_parity import _compare_records, _encode_gpu  # noqa: E402

DEC_TOL = 2e-3


def _params(sets, with_inverse):
    pk0, pv0 = sets[0]
    return kvtc.kv_params_from_arrays(
        np.stack([s[0].T for s in sets]), np.stack([s[0].mu for s in sets]), np.stack([s[0].sigma for s in sets]),
        np.stack([s[0].widths for s in sets]), pk0.r_words,
        np.stack([s[1].T for s in sets]), np.stack([s[1].mu for s in sets]), np.stack([s[1].sigma for s in sets]),
        np.stack([s[1].widths for s in sets]), pv0.r_words,
        T_inv_k=np.stack([s[0].T_inv for s in sets]) if with_inverse else None).upload()


@pytest.mark.parametrize("kind", ["attention_aware", "whitened"])
@pytest.mark.parametrize("name,bits", [("llama_decode_32k", 2.75), ("qwen_batched_8k", 3.0)])
def test_key_transform_encode_and_decode_match_oracle(kind, name, bits):
    w = synth.WORKLOADS[name]
    B = 2 if w.calib == "own_prefix" else 1
    T, T_cap = 1000, 1024
    L = synth.make_layer(w, T=T, steps=1, B=B)
    opt = {"attention_aware_keys": True} if kind == "attention_aware" else {"whitened_keys": True}
    sets = [O.calibrate(ck, cv, cq, bits, bits, **opt) for ck, cv, cq in zip(L.calib_k, L.calib_v, L.calib_q)]
    if kind == "whitened":
        assert all(s[0].T_inv is not None for s in sets)
    P = _params(sets, kind == "whitened")
    per_seq = L.per_seq_params
    k, v = synth.as_float(L.k), synth.as_float(L.v)
    # encode (the tensor-core prefill: bf16, 1000 tokens) against the oracle's records, every entry
    ork, orv = G.oracle_cache(k, v, sets, per_seq, T_cap)
    rk, rv = _encode_gpu(P, L.k, L.v, per_seq, T_cap=T_cap)
    n_diff, n_all = 0.0, 0
    for b in range(B):
        for h in range(w.Hkv):
            pk, pv = sets[G.set_index(b, h, w.Hkv, per_seq)]
            for got, ref, p in ((rk[b, h], ork[b, h], pk), (rv[b, h], orv[b, h], pv)):
                nd, na = _compare_records(got, ref, p, T)
                n_diff += nd
                n_all += na
    assert n_diff / n_all <= 1e-4, (n_diff / n_all, n_all)
    # decode over the oracle's records, ragged lengths
    seq = [T, 617][:B]
    got = G.run_decode(P, ork, orv, L.q[0], seq, w.Hq, per_seq)
    ref = G.oracle_decode(ork, orv, L.q[0], seq, sets, w.Hq, per_seq)
    err = G.rel_l2_rows(got, ref)
    assert err.max() <= DEC_TOL, err.max()


def test_whitened_keys_need_the_inverse():
    """Without the inverse the library takes the non-orthogonal T as orthogonal (k^ = T^T y^): the decode then
    leaves the oracle's result, which shows the inverse is what the decode uses."""
    w = synth.WORKLOADS["llama_decode_32k"]
    T, T_cap = 600, 608
    L = synth.make_layer(w, T=T, steps=1)
    sets = [O.calibrate(ck, cv, cq, 2.75, 2.75, whitened_keys=True)
            for ck, cv, cq in zip(L.calib_k, L.calib_v, L.calib_q)]
    k, v = synth.as_float(L.k), synth.as_float(L.v)
    ork, orv = G.oracle_cache(k, v, sets, False, T_cap)
    ref = G.oracle_decode(ork, orv, L.q[0], [T], sets, w.Hq, False)
    good = G.rel_l2_rows(G.run_decode(_params(sets, True), ork, orv, L.q[0], [T], w.Hq, False), ref)
    bad = G.rel_l2_rows(G.run_decode(_params(sets, False), ork, orv, L.q[0], [T], w.Hq, False), ref)
    assert good.max() <= DEC_TOL
    assert not np.all(bad <= 10 * DEC_TOL)  # (NaN counts as far off)
