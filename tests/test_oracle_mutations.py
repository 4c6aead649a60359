"""Plant a plausible mistake in the CPU oracle (on the CPU, via monkeypatch) and check that a pin catches
it: evidence that the pins constrain every step of the oracle, not just its happy path."""
import numpy as np
import pytest

import oracle_pins as P
from oracle import kvtc_oracle as O

_orig = {name: getattr(O, name) for name in
         ["klt", "key_weights", "calib_statistics", "water_fill_continuous", "water_fill_integer",
          "quantize", "pack", "dequantize", "rotate", "reconstruct", "attention", "half_rn_sat",
          "slot_layout", "fit_layout", "token_slot_layout", "fit_token_layout", "storage_order", "attend_decode",
          "exchange_rate", "joint_split", "attention_aware_key_basis", "whitened_key_transform", "rotary_embed",
          "token_weights", "token_keep", "compact"]}


def _klt_transposed(sigma):
    lam, u = _orig["klt"](sigma)
    return lam, u.T.copy()


def _klt_no_sign_fix(sigma):
    lam, u = np.linalg.eigh(np.asarray(sigma, np.float64))
    o = np.argsort(-lam)
    return lam[o], -u[:, o]


def _key_weights_rows(u, m_q):
    u = np.asarray(u, np.float64)
    return np.einsum("ij,jk,ik->i", u, m_q, u)


def _stats_uncentred(k, v, q):
    mu_k, _, mu_v, _, m_q = _orig["calib_statistics"](k, v, q)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    return mu_k, k.T @ k / len(k), mu_v, v.T @ v / len(v), m_q


def _wf_natural_log(lam, budget, max_bits, iters=200):
    lam = np.asarray(lam, np.float64)
    pos = lam > 0
    if budget <= 0 or not pos.any() or budget >= max_bits * pos.sum():
        return _orig["water_fill_continuous"](lam, budget, max_bits, iters)
    l = np.full(len(lam), -np.inf)
    l[pos] = np.log(lam[pos])
    lo, hi = l[pos].min() - 40, l[pos].max()
    f = lambda t: np.clip(0.5 * (l - t), 0, max_bits)
    for _ in range(iters):
        mid = 0.5 * (lo + hi)
        lo, hi = (mid, hi) if f(mid).sum() > budget else (lo, mid)
    return f(0.5 * (lo + hi)), np.exp(0.5 * (lo + hi))


def _wi_ties_to_smaller(lam, budget, max_bits):
    lam = np.asarray(lam, np.float64)
    br, _ = O.water_fill_continuous(lam, budget, max_bits)
    bi = np.floor(br).astype(np.int64)
    key = np.rint((br - bi) * 1e9)
    cand = sorted([i for i in range(len(lam)) if bi[i] < max_bits and lam[i] > 0],
                  key=lambda i: (-key[i], lam[i], i))
    for i in cand[:int(budget - bi.sum())]:
        bi[i] += 1
    return bi


def _quantize_zero_from_max(y32, p):
    z, s, c = _orig["quantize"](y32, p)
    nz = p.widths > 0
    yp = (np.asarray(y32, np.float32)[:, nz] - p.mu[nz]) * p.inv_sigma[nz]
    return O.half_rn_sat(yp.max(1)), s, c


def _quantize_half_scale(y32, p):
    q = O.TensorParams(p.T, p.mu, p.sigma, np.maximum(p.widths - 1, 0), p.r_words)
    z, s, c = _orig["quantize"](y32, q)
    return z, s, c


def _pack_one_word_late(z16, s16, codes, p):
    rec = _orig["pack"](z16, s16, codes, p)
    out = np.zeros_like(rec)
    out[:, 0] = rec[:, 0]
    out[:, 2:] = rec[:, 1:-1]
    return out


def _pack_msb_first(z16, s16, codes, p):
    rec = _orig["pack"](z16, s16, codes, p)
    out = rec.copy()
    for w in range(1, rec.shape[1]):
        x = rec[:, w].astype(np.uint64)
        r = np.zeros_like(x)
        for b in range(32):
            r |= ((x >> np.uint64(b)) & np.uint64(1)) << np.uint64(31 - b)
        out[:, w] = r.astype(np.uint32)
    return out


def _dequant_no_half(z16, s16, codes, p):
    return _orig["dequantize"](z16, s16, np.asarray(codes) - 0.5, p)


def _rotate_transposed(x, p):
    return (np.asarray(x, np.float64) @ p.T.astype(np.float64)).astype(np.float32)


def _reconstruct_transposed(rec, p):
    y = O.dequantize(*O.unpack(rec, p), p)
    return y @ p.T.astype(np.float64).T


def _attention_unscaled(q, k, v, scale):
    return _orig["attention"](q, k, v, 1.0)


def _half_truncate(x):
    x = np.clip(np.asarray(x, np.float32), -65504, 65504)
    h = x.astype(np.float16)
    over = np.abs(h.astype(np.float32)) > np.abs(x)
    return np.where(over, np.nextafter(h, np.float16(0)), h).astype(np.float16)


def _slot_layout_next_fit(widths, r_words):
    """Never returns to an earlier code word."""
    w = np.asarray(widths, np.int64)
    if w.shape[0] % 2:
        w = np.concatenate([w, [0]])
    word = np.full(w.shape[0] // 2, -1, np.int64)
    pos = np.full(w.shape[0] // 2, -1, np.int64)
    u, used = 0, 0
    for k in range(w.shape[0] // 2):
        sw = int(max(w[2 * k], w[2 * k + 1]))
        if sw == 0:
            continue
        if used + sw > 16:
            u, used = u + 1, 0
        if u >= r_words - 1:
            return None
        word[k], pos[k] = u, used
        used += sw
    return word, pos


def _fit_ties_to_earlier(widths, importance, r_words):
    b = np.asarray(widths, np.int64)
    lam = np.asarray(importance, np.float64)
    w = [int(max(b[2 * k], b[2 * k + 1])) for k in range(len(b) // 2)]
    plam = [float(lam[2 * k] + lam[2 * k + 1]) for k in range(len(b) // 2)]
    while O.slot_layout(np.repeat(w, 2), r_words) is None:
        _, k = min((O.fit_cost_key(plam[k], w[k]), k) for k in range(len(w)) if w[k] > 0)
        w[k] -= 1
    return np.repeat(np.asarray(w, np.int64), 2)


def _fit_cost_ignores_width(widths, importance, r_words):
    b = np.asarray(widths, np.int64)
    lam = np.asarray(importance, np.float64)
    w = [int(max(b[2 * k], b[2 * k + 1])) for k in range(len(b) // 2)]
    plam = [float(lam[2 * k] + lam[2 * k + 1]) for k in range(len(b) // 2)]
    while O.slot_layout(np.repeat(w, 2), r_words) is None:
        _, negk = min((plam[k], -k) for k in range(len(w)) if w[k] > 0)
        w[-negk] -= 1
    return np.repeat(np.asarray(w, np.int64), 2)


def _fit_no_promotion(widths, importance, r_words):
    f = _orig["fit_layout"](widths, importance, r_words)
    b = np.asarray(widths, np.int64)
    return np.minimum(f, b)


def _token_layout_next_fit(widths, r_words):
    w = np.asarray(widths, np.int64)
    word = np.full(w.shape[0], -1, np.int64)
    pos = np.full(w.shape[0], -1, np.int64)
    u, used = 0, 0
    for j in range(w.shape[0]):
        b = int(w[j])
        if b == 0:
            continue
        if used + b > 16:
            u, used = u + 1, 0
        if u >= 2 * r_words - 2:
            return None
        word[j], pos[j] = u, used
        used += b
    return word, pos


def _token_fit_ties_to_earlier(widths, importance, r_words):
    w = [int(x) for x in np.asarray(widths, np.int64)]
    lam = [float(x) for x in np.asarray(importance, np.float64)]
    while O.token_slot_layout(w, r_words) is None:
        _, j = min((O.fit_cost_key(lam[j], w[j]), j) for j in range(len(w)) if w[j] > 0)
        w[j] -= 1
    return np.asarray(w, np.int64)


def _token_pack_swapped_halves(z16, s16, codes, p):
    rec = _orig["pack"](z16, s16, codes, p)
    if p.pairing != "tokens":
        return rec
    out = rec.copy()
    for w in range(2, rec.shape[1]):
        x = rec[:, w].astype(np.uint64)
        out[:, w] = (((x & np.uint64(0xFFFF)) << np.uint64(16)) | (x >> np.uint64(16))).astype(np.uint32)
    return out


def _storage_ties_ascending(widths, lam):
    return sorted(range(len(widths)), key=lambda i: (-int(widths[i]), float(lam[i]), i))


def _attend_ignores_length(q, rec_k, rec_v, pk, pv, seq_len, scale):
    return _orig["attend_decode"](q, rec_k, rec_v, pk, pv, len(rec_k), scale)


def _attend_one_token_short(q, rec_k, rec_v, pk, pv, seq_len, scale):
    return _orig["attend_decode"](q, rec_k, rec_v, pk, pv, max(1, seq_len - 1), scale)


def _rate_alpha_not_squared(lam_v, d):
    return float(np.sum(np.maximum(np.asarray(lam_v, np.float64), 0.0))) / np.sqrt(d)


def _split_ignores_rho(per_set, r_total, rwk_sep, max_bits, d):
    return _orig["joint_split"]([(ik, iv, 1.0) for ik, iv, _ in per_set], r_total, rwk_sep, max_bits, d)


def _aware_ignores_queries(sigma_k, m_q, u0, sweeps=8, grid=48):
    return _orig["attention_aware_key_basis"](sigma_k, np.eye(np.asarray(sigma_k).shape[0]), u0, sweeps, grid)


def _aware_rotates_u_backwards(sigma_k, m_q, u0, sweeps=8, grid=48):
    """Tracks the rotated matrices correctly but turns the basis the other way."""
    A = np.array(sigma_k, np.float64) + np.eye(len(sigma_k)) * (1e-12 * np.trace(sigma_k) / len(sigma_k))
    B = np.array(m_q, np.float64) + np.eye(len(m_q)) * (1e-12 * np.trace(m_q) / len(m_q))
    U = np.array(u0, np.float64)
    a, b = U.T @ A @ U, U.T @ B @ U
    phis = -np.pi / 4 + np.arange(grid) * (np.pi / 2 / grid)
    c, s = np.cos(phis), np.sin(phis)
    d = len(A)
    for _ in range(sweeps):
        for i in range(d - 1):
            for j in range(i + 1, d):
                f = (np.log(c * c * a[i, i] + 2 * c * s * a[i, j] + s * s * a[j, j]) +
                     np.log(s * s * a[i, i] - 2 * c * s * a[i, j] + c * c * a[j, j]) +
                     np.log(c * c * b[i, i] + 2 * c * s * b[i, j] + s * s * b[j, j]) +
                     np.log(s * s * b[i, i] - 2 * c * s * b[i, j] + c * c * b[j, j]))
                k = int(np.argmin(f))
                if not f[k] < f[grid // 2] - 1e-10:
                    continue
                R = np.array([[c[k], -s[k]], [s[k], c[k]]])
                U[:, [i, j]] = U[:, [i, j]] @ R.T
                for M in (a, b):
                    M[:, [i, j]] = M[:, [i, j]] @ R
                    M[[i, j], :] = R.T @ M[[i, j], :]
    return U


def _whitened_full_power(sigma_k, m_q):
    """Whitens with M_Q instead of its square root."""
    A = np.asarray(sigma_k, np.float64)
    M = np.array(m_q, np.float64) + np.eye(len(m_q)) * (1e-12 * np.trace(m_q) / len(m_q))
    lam, V = O.klt(M @ A @ M)
    T = V.T @ M
    T_inv = np.linalg.inv(T)
    c = float(np.linalg.norm(T_inv, axis=0).max())
    return lam * c * c, T * c, T_inv / c


def _whitened_ignores_queries(sigma_k, m_q):
    return _orig["whitened_key_transform"](sigma_k, np.eye(len(m_q)))


def _rope_interleaved(x, pos, base):
    """Pairs (2i, 2i + 1) instead of (i, i + d/2)."""
    x = np.asarray(x, np.float64)
    d = x.shape[-1]
    freq = np.array([float(base) ** (-2.0 * i / d) for i in range(d // 2)])
    c, s = np.cos(pos * freq), np.sin(pos * freq)
    a, b = x[..., 0::2], x[..., 1::2]
    y = np.empty_like(x)
    y[..., 0::2], y[..., 1::2] = a * c - b * s, a * s + b * c
    return y


def _rope_backwards(x, pos, base):
    return _orig["rotary_embed"](x, -pos, base)


def _rope_frequency_halved(x, pos, base):
    """Exponent -i/d instead of -2i/d."""
    return _orig["rotary_embed"](x, pos, np.sqrt(base))


def _weights_first_power(q_obs, k, scale):
    """sum_q p_qt instead of sum_q p_qt^2."""
    q = np.asarray(q_obs, np.float64)
    lg = scale * (q @ np.asarray(k, np.float64).T)
    p = np.exp(lg - lg.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    return p.sum(axis=0) / np.sqrt(q.shape[0])


def _keep_ties_to_later(lam, keep):
    lam = np.asarray(lam, np.float64)
    order = sorted(range(lam.shape[0]), key=lambda t: (-lam[t], -t))
    return np.array(sorted(order[:keep]), np.int64)


def _compact_keeps_pairs(rec, p, keep_idx):
    """Copies whole value records (the kept token's partner comes along) instead of re-pairing tokens."""
    if p.pairing == "channels":
        return _orig["compact"](rec, p, keep_idx)
    return np.asarray(rec)[np.asarray(keep_idx) // 2]


MUTATIONS = [
    ("klt", _klt_transposed, P.pin_klt_known_spectrum),
    ("klt", _klt_no_sign_fix, P.pin_klt_known_spectrum),
    ("key_weights", _key_weights_rows, P.pin_key_distortion_monte_carlo),
    ("calib_statistics", _stats_uncentred, P.pin_statistics_closed_form),
    ("water_fill_continuous", _wf_natural_log, P.pin_water_fill_golden),
    ("water_fill_integer", _wi_ties_to_smaller, P.pin_water_fill_golden),
    ("quantize", _quantize_zero_from_max, P.pin_quantize_pack_golden),
    ("quantize", _quantize_half_scale, P.pin_quantize_pack_golden),
    ("pack", _pack_one_word_late, P.pin_quantize_pack_golden),
    ("pack", _pack_msb_first, P.pin_quantize_pack_golden),
    ("dequantize", _dequant_no_half, P.pin_quantizer_error_bound),
    ("rotate", _rotate_transposed, P.pin_sixteen_bits_preserve_attention),
    ("reconstruct", _reconstruct_transposed, P.pin_decode_brute_force),
    ("attention", _attention_unscaled, P.pin_decode_brute_force),
    ("half_rn_sat", _half_truncate, P.pin_half_conversion),
    ("slot_layout", _slot_layout_next_fit, P.pin_layout_fit_golden),
    ("fit_layout", _fit_ties_to_earlier, P.pin_layout_fit_golden),
    ("fit_layout", _fit_cost_ignores_width, P.pin_layout_fit_golden),
    ("fit_layout", _fit_no_promotion, P.pin_layout_fit_golden),
    ("token_slot_layout", _token_layout_next_fit, P.pin_token_layout_fit_golden),
    ("fit_token_layout", _token_fit_ties_to_earlier, P.pin_token_layout_fit_golden),
    ("pack", _token_pack_swapped_halves, P.pin_token_pack_golden),
    ("storage_order", _storage_ties_ascending, P.pin_storage_order),
    ("attend_decode", _attend_ignores_length, P.pin_decode_brute_force),
    ("attend_decode", _attend_one_token_short, P.pin_decode_brute_force),
    ("exchange_rate", _rate_alpha_not_squared, P.pin_exchange_rate_monte_carlo),
    ("joint_split", _split_ignores_rho, P.pin_joint_split_by_enumeration),
    ("attention_aware_key_basis", _aware_ignores_queries, P.pin_aware_basis_bounds),
    ("attention_aware_key_basis", _aware_rotates_u_backwards, P.pin_aware_basis_two_channels),
    ("whitened_key_transform", _whitened_full_power, P.pin_whitened_key_transform),
    ("whitened_key_transform", _whitened_ignores_queries, P.pin_whitened_key_transform),
    ("rotary_embed", _rope_interleaved, P.pin_rotary_embedding),
    ("rotary_embed", _rope_backwards, P.pin_rotary_embedding),
    ("rotary_embed", _rope_frequency_halved, P.pin_rotary_embedding),
    ("token_weights", _weights_first_power, P.pin_token_weights),
    ("token_keep", _keep_ties_to_later, P.pin_token_keep),
    ("compact", _compact_keeps_pairs, P.pin_compact),
]


@pytest.mark.parametrize("name,mutant,pin", MUTATIONS, ids=[f"{m[0]}:{m[1].__name__}" for m in MUTATIONS])
def test_pin_catches_planted_mistake(monkeypatch, name, mutant, pin):
    monkeypatch.setattr(O, name, mutant)
    with pytest.raises(AssertionError):
        pin()
