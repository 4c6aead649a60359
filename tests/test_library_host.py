"""C-ABI library on the CPU: exported symbols, host calibration against the oracle, persistence and argument
errors. No compute kernel is launched here."""
import math
import os
import subprocess

import numpy as np
import pytest

from oracle import kvtc_oracle as O
from transform_coded_kv_02_b300 import kvtc, synth

from conftest import read_golden


def test_library_exports_every_declared_symbol():
    out = subprocess.run(["nm", "-D", "--defined-only", kvtc.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    syms = {line.split()[-1] for line in out.splitlines() if line.strip()}
    declared = kvtc.exported_symbols()
    assert len(declared) >= 25
    missing = [s for s in declared if s not in syms]
    assert not missing, missing
    for s in declared:  # and they resolve through the dynamic loader
        assert getattr(kvtc._lib, s) is not None


def test_water_fill_golden_library():
    for lam, C, bmax, b_real, b_int in read_golden("water_fill_small.txt"):
        lam = np.array([float(x) for x in lam.split()])
        got = kvtc.kv_debug_water_fill(lam, int(C), int(bmax))
        assert got.tolist() == [int(x) for x in b_int.split()]


def test_water_fill_library_matches_oracle():
    rng = np.random.default_rng(21)
    for trial in range(200):
        d = int(rng.integers(1, 129))
        lam = np.exp(rng.normal(0, 3, d))
        lam[rng.random(d) < 0.05] = 0.0
        if trial % 7 == 0:
            lam = np.round(lam)  # ties
        C = int(rng.integers(0, 8 * d + 8))
        assert np.array_equal(kvtc.kv_debug_water_fill(lam, C, 8), O.water_fill_integer(lam, C, 8)), trial


def test_jacobi_eigensolver_against_lapack():
    rng = np.random.default_rng(22)
    for d in (2, 5, 32, 128):
        Q = synth.random_orthogonal(d, rng)
        lam = np.exp(rng.normal(0, 2, d))
        S = (Q * lam) @ Q.T
        ev, vec = kvtc.kv_debug_eigh(S)
        le, _ = np.linalg.eigh(S)
        assert np.allclose(ev, np.sort(le)[::-1], rtol=1e-10, atol=1e-13 * lam.max())
        assert np.linalg.norm(vec.T @ vec - np.eye(d)) < 1e-12 * d
        assert np.linalg.norm((vec * ev) @ vec.T - S) < 1e-11 * np.linalg.norm(S)
        lo, uo = O.klt(S)
        for i in range(d):  # same sign convention -> same vectors for distinct eigenvalues
            assert np.allclose(vec[:, i], uo[:, i], atol=1e-8)


@pytest.mark.parametrize("name", ["tiny", "qwen_batched_8k"])
def test_host_calibration_matches_oracle(name):
    w = synth.WORKLOADS[name]
    L = synth.make_layer(w, T=256 if name != "tiny" else 64, B=2 if name != "tiny" else 1, steps=1)
    bits = w.bits[0]
    sets = list(zip(L.calib_k, L.calib_v, L.calib_q))
    P = kvtc.kv_calibrate(sets, bits, bits)
    assert P.num_sets == len(sets)
    for s, (ck, cv, cq) in enumerate(sets):
        pk, pv = O.calibrate(ck, cv, cq, bits, bits)
        for t, po in ((0, pk), (1, pv)):
            info = P.info(s, t)
            assert info["r_words"] == po.r_words
            assert np.array_equal(info["widths"], po.widths)
            assert np.allclose(info["eigvals"], po.eigvals, rtol=1e-9, atol=1e-12 * po.eigvals.max())
            # rows of T: same channels in the same order, same sign (non-degenerate spectra)
            assert np.max(np.abs(info["T"].astype(np.float64) - po.T.astype(np.float64))) < 1e-5
            assert np.allclose(info["mu"], po.mu, atol=1e-5)
            assert np.allclose(info["sigma"], po.sigma, rtol=1e-6)
            if t == 0:
                assert np.allclose(info["importance"], po.importance, rtol=1e-8)


@pytest.mark.parametrize("name,bits", [("llama_decode_32k", 2.75), ("llama_long_128k", 1.33), ("qwen_batched_8k", 3.0)])
def test_host_joint_calibration_matches_oracle(name, bits):
    """The joint key/value split: the library picks the oracle's split for the table, then allocates and lays
    out each tensor as the oracle does."""
    w = synth.WORKLOADS[name]
    # sequences calibrated on their own prefix need more tokens than channels for a full-rank covariance
    # (unique eigenvectors)
    L = synth.make_layer(w, T=256, B=2 if w.calib == "own_prefix" else 1, steps=1)
    sets = list(zip(L.calib_k, L.calib_v, L.calib_q))
    P = kvtc.kv_calibrate(sets, bits, bits, joint=True)
    ref = O.calibrate_joint(sets, bits, bits)
    assert P.record_words(0) + P.record_words(1) == 2 * O.record_words(bits, 128)
    for s, (pk, pv) in enumerate(ref):
        for t, po in ((0, pk), (1, pv)):
            info = P.info(s, t)
            assert info["r_words"] == po.r_words
            assert np.array_equal(info["widths"], po.widths)
            assert np.max(np.abs(info["T"].astype(np.float64) - po.T.astype(np.float64))) < 1e-5


@pytest.mark.parametrize("name", ["tiny", "llama_decode_32k", "qwen_batched_8k"])
def test_host_attention_aware_key_basis_matches_oracle(name):
    """The attention-aware key basis: the library's Jacobi sweeps take the oracle's rotations (same grid, same
    order, same threshold), so the transforms, variances and widths agree; the value side is untouched."""
    w = synth.WORKLOADS[name]
    L = synth.make_layer(w, T=256, B=2 if w.calib == "own_prefix" else 1, steps=1)
    sets = list(zip(L.calib_k, L.calib_v, L.calib_q))[:3]
    bits = w.bits[0]
    P = kvtc.kv_calibrate(sets, bits, bits, attention_aware_keys=True)
    for s, (ck, cv, cq) in enumerate(sets):
        pk, pv = O.calibrate(ck, cv, cq, bits, bits, attention_aware_keys=True)
        for t, po in ((0, pk), (1, pv)):
            info = P.info(s, t)
            assert np.array_equal(info["widths"], po.widths)
            assert np.max(np.abs(info["T"].astype(np.float64) - po.T.astype(np.float64))) < 1e-5
            assert np.allclose(info["eigvals"], po.eigvals, rtol=1e-9, atol=1e-12 * np.abs(po.eigvals).max())


def test_host_both_calibration_options_match_oracle():
    """The attention-aware key basis and the joint split together: the library's split, widths and transforms
    are the oracle's."""
    w = synth.WORKLOADS["llama_decode_32k"]
    L = synth.make_layer(w, T=256, steps=1)
    sets = list(zip(L.calib_k, L.calib_v, L.calib_q))[:3]
    P = kvtc.kv_calibrate(sets, 2.75, 2.75, joint=True, attention_aware_keys=True)
    ref = O.calibrate_joint(sets, 2.75, 2.75, attention_aware_keys=True)
    assert (P.record_words(0), P.record_words(1)) == (ref[0][0].r_words, ref[0][1].r_words) == (14, 8)
    for s, (pk, pv) in enumerate(ref):
        for t, po in ((0, pk), (1, pv)):
            info = P.info(s, t)
            assert np.array_equal(info["widths"], po.widths)
            assert np.max(np.abs(info["T"].astype(np.float64) - po.T.astype(np.float64))) < 1e-5


def test_key_basis_flag_is_checked():
    L = synth.make_layer(synth.WORKLOADS["tiny"], T=16, steps=1)
    with pytest.raises(kvtc.KvError) as e:
        kvtc.kv_calibrate(list(zip(L.calib_k, L.calib_v, L.calib_q)), 2.75, 2.75, attention_aware_keys=3)
    assert e.value.status == kvtc.KV_ERR_INVALID_ARG


@pytest.mark.parametrize("name", ["tiny", "llama_decode_32k", "qwen_batched_8k"])
def test_host_whitened_key_transform_matches_oracle(name):
    """key_basis 2, the non-orthogonal key transform: the library's two Jacobi eigendecompositions give the
    oracle's transform, its inverse (kept beside it in storage order), variances and widths; values untouched."""
    w = synth.WORKLOADS[name]
    L = synth.make_layer(w, T=256, B=2 if w.calib == "own_prefix" else 1, steps=1)
    sets = list(zip(L.calib_k, L.calib_v, L.calib_q))[:3]
    bits = w.bits[0]
    P = kvtc.kv_calibrate(sets, bits, bits, whitened_keys=True)
    for s, (ck, cv, cq) in enumerate(sets):
        pk, pv = O.calibrate(ck, cv, cq, bits, bits, whitened_keys=True)
        info = P.info(s, 0)
        assert np.array_equal(info["widths"], pk.widths)
        scale = np.abs(pk.T).max()
        assert np.max(np.abs(info["T"].astype(np.float64) - pk.T)) < 1e-5 * scale
        ti = P.inverse(s, 0)
        assert ti is not None
        assert np.max(np.abs(ti.astype(np.float64) - pk.T_inv)) < 1e-5 * np.abs(pk.T_inv).max()
        assert np.allclose(info["eigvals"], pk.eigvals, rtol=1e-6, atol=1e-12 * np.abs(pk.eigvals).max())
        # the inverse undoes the transform; every column of it has norm <= 1 (the decode's q' scale bound)
        assert np.max(np.abs(ti.astype(np.float64) @ info["T"].astype(np.float64) - np.eye(128))) < 1e-4
        assert np.linalg.norm(ti.astype(np.float64), axis=0).max() <= 1 + 1e-6
        assert P.inverse(s, 1) is None
        assert np.array_equal(P.info(s, 1)["widths"], pv.widths)


def test_params_inverse_survives_save_and_load(tmp_path):
    """A table with a non-orthogonal key transform keeps its inverse through kv_params_save / kv_params_load;
    kv_params_set_inverse(None) removes it."""
    w = synth.WORKLOADS["tiny"]
    L = synth.make_layer(w, T=256, steps=1)
    P = kvtc.kv_calibrate(list(zip(L.calib_k, L.calib_v, L.calib_q)), 2.75, 2.75, whitened_keys=True)
    path = tmp_path / "whitened.kvtc"
    P.save(str(path))
    Q = kvtc.kv_params_load(str(path))
    assert np.array_equal(Q.inverse(0, 0), P.inverse(0, 0))
    assert Q.inverse(0, 1) is None
    Q.set_inverse(0, None)
    assert Q.inverse(0, 0) is None


def test_joint_flag_is_checked():
    L = synth.make_layer(synth.WORKLOADS["tiny"], T=16, steps=1)
    sets = list(zip(L.calib_k, L.calib_v, L.calib_q))
    with pytest.raises(kvtc.KvError) as e:
        kvtc.kv_calibrate(sets, 2.75, 2.75, joint=2)
    assert e.value.status == kvtc.KV_ERR_INVALID_ARG


def test_params_save_load_roundtrip(tmp_path):
    L = synth.make_layer(synth.WORKLOADS["tiny"], T=16, steps=1)
    P = kvtc.kv_calibrate(list(zip(L.calib_k, L.calib_v, L.calib_q)), 2.75, 2.75)
    path = str(tmp_path / "p.kvtc")
    P.save(path)
    Q = kvtc.kv_params_load(path)
    for t in (0, 1):
        a, b = P.info(0, t), Q.info(0, t)
        for key in a:
            assert np.array_equal(np.asarray(a[key]), np.asarray(b[key])), key
    raw = bytearray(open(path, "rb").read())
    raw[100] ^= 0x40
    open(path, "wb").write(bytes(raw))
    with pytest.raises(kvtc.KvError) as e:
        kvtc.kv_params_load(path)
    assert e.value.status == kvtc.KV_ERR_IO
    open(path, "wb").write(bytes(raw[:50]))
    with pytest.raises(kvtc.KvError) as e:
        kvtc.kv_params_load(path)
    assert e.value.status == kvtc.KV_ERR_IO
    with pytest.raises(kvtc.KvError) as e:
        kvtc.kv_params_load(str(tmp_path / "missing"))
    assert e.value.status == kvtc.KV_ERR_IO


def test_params_save_load_unequal_record_lengths(tmp_path):
    """A table from the joint split (14 key and 8 value words on the Llama-shaped statistics) keeps both
    record lengths and every array through save and load."""
    L = synth.make_layer(synth.WORKLOADS["llama_decode_32k"], T=16, steps=1)
    sets = list(zip(L.calib_k, L.calib_v, L.calib_q))[:2]
    P = kvtc.kv_calibrate(sets, 2.75, 2.75, joint=True, attention_aware_keys=True)
    assert (P.record_words(0), P.record_words(1)) == (14, 8)
    path = str(tmp_path / "joint.kvtc")
    P.save(path)
    Q = kvtc.kv_params_load(path)
    assert (Q.record_words(0), Q.record_words(1)) == (14, 8)
    for s in range(2):
        for t in (0, 1):
            a, b = P.info(s, t), Q.info(s, t)
            for key in a:
                assert np.array_equal(np.asarray(a[key]), np.asarray(b[key])), (s, t, key)


def test_calibrate_argument_errors():
    rng = np.random.default_rng(0)
    k = rng.normal(size=(64, 128)).astype(np.float32)
    with pytest.raises(kvtc.KvError) as e:
        kvtc.kv_calibrate([(k, k, k)], 2.75, 2.75, d=64)
    assert e.value.status == kvtc.KV_ERR_UNSUPPORTED
    with pytest.raises(kvtc.KvError) as e:
        kvtc.kv_calibrate([(k, k, k)], 8.5, 2.75)
    assert e.value.status == kvtc.KV_ERR_BUDGET
    with pytest.raises(kvtc.KvError) as e:
        kvtc.kv_calibrate([(k, k, k)], 0.1, 2.75)
    assert e.value.status == kvtc.KV_ERR_BUDGET
    bad = k.copy()
    bad[3, 7] = np.nan
    with pytest.raises(kvtc.KvError) as e:
        kvtc.kv_calibrate([(k, bad, k)], 2.75, 2.75)
    assert e.value.status == kvtc.KV_ERR_NUMERIC
    with pytest.raises(kvtc.KvError) as e:
        kvtc.kv_calibrate([(k[:1], k[:1], k)], 2.75, 2.75)
    assert e.value.status == kvtc.KV_ERR_INVALID_ARG


def test_params_from_arrays_validation():
    d = 128
    T = np.eye(d, dtype=np.float32)[None]
    mu = np.zeros((1, d), np.float32)
    sg = np.ones((1, d), np.float32)
    w = np.zeros((1, d), np.int32)
    w[0, :40] = 8
    with pytest.raises(kvtc.KvError) as e:  # 320 bits > 10 words of codes
        kvtc.kv_params_from_arrays(T, mu, sg, w, 10, T, mu, sg, w, 11)
    assert e.value.status == kvtc.KV_ERR_BUDGET
    w2 = np.zeros((1, d), np.int32)
    w2[0, :48] = 6  # 288 bits fit the budget, but 24 six-bit slots need 12 code words (2 per word)
    with pytest.raises(kvtc.KvError) as e:
        kvtc.kv_params_from_arrays(T, mu, sg, w2, 11, T, mu, sg, w2, 11)
    assert e.value.status == kvtc.KV_ERR_BUDGET
    w3 = np.zeros((1, d), np.int32)
    w3[0, 5] = 9  # wider than 8 bits
    with pytest.raises(kvtc.KvError) as e:
        kvtc.kv_params_from_arrays(T, mu, sg, w3, 11, T, mu, sg, w3, 11)
    assert e.value.status == kvtc.KV_ERR_INVALID_ARG
    w4 = np.zeros((1, d), np.int32)
    w4[0, 5] = 3  # zero-width channels before a nonzero one are allowed (a pair may lose all its bits)
    kvtc.kv_params_from_arrays(T, mu, sg, w4, 11, T, mu, sg, w4, 11)
    P = kvtc.kv_params_from_arrays(T, mu, sg, w, 11, T, mu, sg, w, 11)
    assert P.record_words(0) == 11 and P.info(0, 0)["widths"].sum() == 320


def test_encode_refuses_params_not_uploaded():
    d = 128
    T = np.eye(d, dtype=np.float32)[None]
    z = np.zeros((1, d), np.float32)
    w = np.zeros((1, d), np.int32)
    P = kvtc.kv_params_from_arrays(T, z, z + 1, w, 1, T, z, z + 1, w, 1)
    cache = kvtc.make_cache(16, 16, 1, 1, 64)
    with pytest.raises(kvtc.KvError) as e:
        kvtc.kv_encode(P, cache, 16, 16, kvtc.KV_DTYPE_BF16, 1, 4, 16, stream=0)
    assert e.value.status == kvtc.KV_ERR_INVALID_ARG
    assert "not uploaded" in str(e.value)


def test_sizes():
    L = synth.make_layer(synth.WORKLOADS["tiny"], T=16, steps=1)
    P = kvtc.kv_calibrate(list(zip(L.calib_k, L.calib_v, L.calib_q)), 2.75, 1.33)
    assert kvtc.kv_cache_bytes(P, 0, 2, 8, 1024) == 2 * 8 * 1024 * 11 * 4
    assert kvtc.kv_cache_bytes(P, 1, 2, 8, 1024) == 2 * 8 * 1024 * 5 * 4


def test_rope_base_is_kept_and_checked(tmp_path):
    """The rotary base set on a table survives save and load (file version 3); negative or non-finite bases are
    refused; 0 removes it."""
    L = synth.make_layer(synth.WORKLOADS["tiny"], T=16, steps=1)
    P = kvtc.kv_calibrate(list(zip(L.calib_k, L.calib_v, L.calib_q)), 2.75, 2.75)
    assert P.rope_base == 0.0
    P.set_rope(500000.0)
    path = str(tmp_path / "rope.kvtc")
    P.save(path)
    assert kvtc.kv_params_load(path).rope_base == 500000.0
    for bad in (-1.0, float("inf"), float("nan")):
        with pytest.raises(kvtc.KvError) as e:
            P.set_rope(bad)
        assert e.value.status == kvtc.KV_ERR_INVALID_ARG
    P.set_rope(0.0)
    P.save(path)
    assert kvtc.kv_params_load(path).rope_base == 0.0


def test_paged_calls_refuse_params_not_uploaded():
    d = 128
    T = np.eye(d, dtype=np.float32)[None]
    z = np.zeros((1, d), np.float32)
    w = np.zeros((1, d), np.int32)
    P = kvtc.kv_params_from_arrays(T, z, z + 1, w, 1, T, z, z + 1, w, 1)
    cache = kvtc.make_paged_cache(16, 16, 4, 32, 1, 1, 1, 4, 16)
    with pytest.raises(kvtc.KvError) as e:
        kvtc.kv_encode_paged(P, cache, 16, 16, kvtc.KV_DTYPE_BF16, 4, 16, stream=0)
    assert e.value.status == kvtc.KV_ERR_INVALID_ARG and "not uploaded" in str(e.value)
    with pytest.raises(kvtc.KvError) as e:
        kvtc.kv_attend_decode_paged(P, cache, 16, 4, 16, None, 0.1, 16, 16, ws_bytes=1 << 20, stream=0)
    assert e.value.status == kvtc.KV_ERR_INVALID_ARG and "not uploaded" in str(e.value)


def test_paged_sizes():
    L = synth.make_layer(synth.WORKLOADS["tiny"], T=16, steps=1)
    P = kvtc.kv_calibrate(list(zip(L.calib_k, L.calib_v, L.calib_q)), 2.75, 1.33)
    assert kvtc.kv_paged_cache_bytes(P, 0, 100, 64, 8) == 100 * 8 * 64 * 11 * 4
    assert kvtc.kv_paged_cache_bytes(P, 1, 100, 64, 8) == 100 * 8 * 64 * 5 * 4
    assert kvtc.kv_paged_cache_bytes(P, 0, 0, 64, 8) == 0
