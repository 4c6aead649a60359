"""The two calibration options beyond the default, measured with the oracle at the same bytes per token on the
Llama-shaped layer (outlier key channels, rotary keys): the joint key/value split of the record moves record
words to the keys, and the attention-aware key basis replaces the KLT; each lowers the decode's error against
exact attention on the unquantised tokens, and together they lower it most."""
import numpy as np

from oracle import kvtc_oracle as O
from transform_coded_kv_02_b300 import synth


def _decode_error(L, sets, w, T, steps):
    k, v = synth.as_float(L.k), synth.as_float(L.v)
    num = den = 0.0
    for h in range(w.Hkv):
        pk, pv = sets[h]
        rk, rv = O.encode(k[0, h], pk), O.encode(v[0, h], pv)
        for s in range(steps):
            q = synth.as_float(L.q[s, 0, h * w.g:(h + 1) * w.g])
            o = O.attend_decode(q, rk, rv, pk, pv, T, 1 / np.sqrt(w.d))
            ex = O.attention(q, k[0, h], v[0, h], 1 / np.sqrt(w.d))
            num += np.sum((o - ex) ** 2)
            den += np.sum(ex ** 2)
    return float(np.sqrt(num / den))


def test_joint_split_lowers_attention_error_llama_shape():
    w = synth.WORKLOADS["llama_decode_32k"]
    T, steps = 1024, 4
    L = synth.make_layer(w, T=T, steps=steps)
    sets_in = list(zip(L.calib_k, L.calib_v, L.calib_q))
    sep = [O.calibrate(k, v, q, 2.75, 2.75) for k, v, q in sets_in]
    jnt = O.calibrate_joint(sets_in, 2.75, 2.75)
    assert (jnt[0][0].r_words, jnt[0][1].r_words) == (14, 8)       # same 22 words per token, keys get more
    e_sep, e_jnt = _decode_error(L, sep, w, T, steps), _decode_error(L, jnt, w, T, steps)
    print("relative L2 error against exact attention: separate %.4f, joint %.4f" % (e_sep, e_jnt))
    assert e_jnt < 0.9 * e_sep


def test_attention_aware_keys_lower_attention_error_llama_shape():
    w = synth.WORKLOADS["llama_decode_32k"]
    T, steps = 1024, 4
    L = synth.make_layer(w, T=T, steps=steps)
    sets_in = list(zip(L.calib_k, L.calib_v, L.calib_q))
    klt = [O.calibrate(k, v, q, 2.75, 2.75) for k, v, q in sets_in]
    aware = [O.calibrate(k, v, q, 2.75, 2.75, attention_aware_keys=True) for k, v, q in sets_in]
    both = O.calibrate_joint(sets_in, 2.75, 2.75, attention_aware_keys=True)
    e_klt, e_aware, e_both = (_decode_error(L, s, w, T, steps) for s in (klt, aware, both))
    print("relative L2 error against exact attention: KLT %.4f, attention-aware keys %.4f, both options %.4f"
          % (e_klt, e_aware, e_both))
    assert e_aware < 0.9 * e_klt and e_both < e_aware


def test_whitened_keys_lower_attention_error_llama_shape():
    """The non-orthogonal key transform (the attention-aware distortion is mean-squared in its domain) against
    the KLT and the attention-aware orthogonal basis, same bytes per token."""
    w = synth.WORKLOADS["llama_decode_32k"]
    T, steps = 1024, 4
    L = synth.make_layer(w, T=T, steps=steps)
    sets_in = list(zip(L.calib_k, L.calib_v, L.calib_q))
    klt = [O.calibrate(k, v, q, 2.75, 2.75) for k, v, q in sets_in]
    white = [O.calibrate(k, v, q, 2.75, 2.75, whitened_keys=True) for k, v, q in sets_in]
    e_klt, e_white = _decode_error(L, klt, w, T, steps), _decode_error(L, white, w, T, steps)
    print("relative L2 error against exact attention: KLT %.4f, whitened keys %.4f" % (e_klt, e_white))
    assert e_white < 0.85 * e_klt


def test_joint_split_keeps_the_qwen_shape_even():
    """On the Qwen-shaped workload (Student-t keys, no outlier channels, one parameter set per sequence) the even
    split measured best at 2, 3 and 4 bits (relative errors 0.096, 0.043, 0.021 against 0.104, 0.046, 0.023 for
    the splits a calibration-measured exchange rate picks); the joint split keeps it there."""
    w = synth.WORKLOADS["qwen_batched_8k"]
    L = synth.make_layer(w, T=1024, B=2, steps=1)
    sets_in = list(zip(L.calib_k, L.calib_v, L.calib_q))
    for bits, rw in ((2.0, 8), (3.0, 12), (4.0, 16)):
        sets = O.calibrate_joint(sets_in, bits, bits)
        assert (sets[0][0].r_words, sets[0][1].r_words) == (rw, rw), bits
